// Device building blocks shared by the libar kernels (sm_103a).
//
// A "pack" is 16 bytes: 8 bf16/fp16 or 4 fp32 elements, the unit of every vector load and
// store (page "[OUTDATED] perf: optimize fused AllReduce + RMSNorm (custom_all_reduce)",
// Technical Details / 2stage: each thread reduces one 16-byte pack across all inputs).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ar {

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

constexpr int kMaxPartials = 8;
constexpr int kPackBytes = 16;

// ---------------------------------------------------------------------------
// kernel parameter blocks (passed by value; the partial pointers travel in them)
// ---------------------------------------------------------------------------
struct ReduceParams {
  const void* x[kMaxPartials];
  void* out;
  int64_t npacks;      // full 16-byte packs
  int64_t numel;       // elements
  int64_t full_tiles;  // npacks / (blockDim * unroll)
  int prefetch;        // 1: warm L2 with the first tile before waiting for the previous grid
};

struct FusedParams {
  const void* x[kMaxPartials];
  const void* res_in;
  void* res_out;
  const void* w;
  void* out;
  uint8_t* q;
  float* scale;
  int64_t m;
  int h;             // elements per row
  int row_packs;     // packs (8 elements) per row, ceil(h / 8)
  int chunk_packs;   // packs per CTA of a cluster (== row_packs without a cluster)
  int csize;         // CTAs per row (cluster size), 1..16
  float eps;
  float inv_h;       // 1 / h
  int gemma;
  int skip_norm;     // 1: no normalisation, y = z (weight unused)
  int out_f32;       // 1: `out` holds fp32 values of y before their rounding
  int group_lanes;   // per-group FP8: lanes (packs) per group, group / 8; 0: per-token FP8
  int ngroups;       // per-group FP8: groups per row, h / group
  int64_t ld_in;     // elements between row starts of the partials and residual_in (0: h)
  int64_t ld_out;    // elements between row starts of residual_out, out and q (0: h)
  int prefetch;      // 1: warm L2 with the first rows' inputs before waiting for the previous grid
};

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------

// Every kernel starts with these two.  griddepcontrol.wait blocks until the grids this
// one depends on (the previous kernels on the stream) have completed and their memory is
// visible, so it must precede the first global read; it returns at once when the launch
// carried no programmatic dependency.  griddepcontrol.launch_dependents then lets the next
// kernel on the stream be scheduled early (once every CTA of this grid has started), so
// its launch latency overlaps this grid's work; the next kernel does its own wait before
// touching memory.
__device__ __forceinline__ void pdl_wait_and_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16) at a 16-byte-aligned global address into L2.
// It moves nothing into the kernel, so it may be issued before griddepcontrol.wait: a line
// that the previous grid writes afterwards is updated in L2, the point of coherence of
// global memory (SM stores write through to it), so later reads still see the new value.
// Issued ahead of the wait, the first DRAM reads of a kernel overlap the tail of the one
// before it on the stream.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// memory access
// ---------------------------------------------------------------------------

// 16-byte streaming load through the non-coherent path without L1 allocation: every
// input element is read exactly once per call.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 16-byte load kept in L1/L2 normally (the weight row, re-read by every row's CTA).
__device__ __forceinline__ uint4 ld_keep(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_u16(const void* p) {
  unsigned short v;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_f32(const void* p) {
  float v;
  asm("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_u16(void* p, uint16_t v) {
  asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

__device__ __forceinline__ void st_u8(void* p, uint8_t v) {
  asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "h"((unsigned short)v) : "memory");
}

__device__ __forceinline__ void st_f32(void* p, float v) {
  asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// ---------------------------------------------------------------------------
// element conversions (hardware cvt, round-to-nearest-even)
// ---------------------------------------------------------------------------

template <int DT>
__device__ __forceinline__ float to_f32(uint32_t bits16);

template <>
__device__ __forceinline__ float to_f32<kBF16>(uint32_t b) {
  return __uint_as_float(b << 16);
}

template <>
__device__ __forceinline__ float to_f32<kF16>(uint32_t b) {
  float f;
  unsigned short h = (unsigned short)b;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}

// Round two floats to the 16-bit type and pack them: `lo` in bits 0..15.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<kBF16>(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <>
__device__ __forceinline__ uint32_t pack2<kF16>(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int DT>
__device__ __forceinline__ uint16_t round1(float v) {
  return (uint16_t)(pack2<DT>(v, 0.0f) & 0xFFFFu);
}

// Unpack the 8 16-bit elements of a pack into floats (element 0 = lowest address).
template <int DT>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = to_f32<DT>(w[i] & 0xFFFFu);
    f[2 * i + 1] = to_f32<DT>(w[i] >> 16);
  }
}

// acc[e] = acc[e] + (float)x_e for the 8 16-bit values x of a pack, with mixed-precision
// adds (a 16-bit operand, an fp32 operand and result): the conversion to fp32 is exact, so
// each sum is the same single fp32 rounding as converting first and adding.
template <int DT>
__device__ __forceinline__ void add8(float (&acc)[8], const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == kBF16)
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
          : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
          : "r"(w[i]));
    else
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
          : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
          : "r"(w[i]));
  }
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  v.x = pack2<DT>(f[0], f[1]);
  v.y = pack2<DT>(f[2], f[3]);
  v.z = pack2<DT>(f[4], f[5]);
  v.w = pack2<DT>(f[6], f[7]);
  return v;
}

// Two fp32 values -> two OCP E4M3 codes, saturating to +-448, round-to-nearest-even;
// `lo` goes to bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Correctly rounded y / d from r = RN(1/d) with one correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q0 = RN(y r) is within an ulp of y / d, the remainder y - q0 d is
// exact through the fused multiply-add, and RN(q0 + rem r) is RN(y / d) when r is the
// correctly rounded reciprocal of a normal d and neither the remainder nor the quotient
// leaves the normal range.  A binary quotient is never exactly half-way between two floats,
// so there are no ties to break.  The correction of a zero quotient would return +0 for
// y = -0 ((+0) + (-0) = +0), so the sign is taken from y, as IEEE division keeps it.
__device__ __forceinline__ float div_rn_by(float y, float d, float r) {
  const float q0 = y * r;
  const float rem = fmaf(-q0, d, y);
  return copysignf(fmaf(rem, r, q0), y);
}

// Smallest row (or group) maximum for which the FP8 quotients take div_rn_by.  With
// amax >= 2^-80: scale = RN(amax / 448) >= 2^-89 is normal and 1 / scale <= 2^89 finite;
// a quotient that can reach a nonzero E4M3 code (|y / scale| >= 2^-10, half the smallest
// subnormal code) has |y| >= 2^-99, so the remainder is a multiple of at least 2^-146 and
// exact; smaller quotients round to code 0 both ways (q0 <= 2^-10 and the correction of a
// quotient below 2^-10 is not positive).  Below this bound (bf16 rows or groups of tiny
// values; an fp16 maximum is at least 2^-24) scale can be subnormal and its reciprocal
// infinite, so each quotient is an IEEE binary32 division instead.
constexpr float kFp8ReciprocalMinAmax = 0x1p-80f;

// How the FP8 codes of one row or group with maximum magnitude `am` are formed.
struct Fp8Scale {
  float scale;  // RN(am / 448), the stored scale
  float rcp;    // RN(1 / scale) when mode == 1
  int mode;     // 0: am == 0, every code 0 (no division); 1: div_rn_by; 2: IEEE division
};

__device__ __forceinline__ Fp8Scale fp8_scale(float am) {
  Fp8Scale s;
  s.scale = __fdiv_rn(am, 448.0f);
  s.mode = am == 0.0f ? 0 : (am >= kFp8ReciprocalMinAmax ? 1 : 2);
  s.rcp = s.mode == 1 ? __frcp_rn(s.scale) : 0.0f;
  return s;
}

// E4M3 codes (saturating, round-to-nearest-even) of y / scale for 8 rounded values y, in
// address order (element 0 in the lowest byte).
__device__ __forceinline__ uint2 fp8_codes8(const float (&y)[8], const Fp8Scale& s) {
  uint32_t c[4] = {0u, 0u, 0u, 0u};
  if (s.mode == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = e4m3x2(div_rn_by(y[2 * i], s.scale, s.rcp), div_rn_by(y[2 * i + 1], s.scale, s.rcp));
  } else if (s.mode == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = e4m3x2(__fdiv_rn(y[2 * i], s.scale), __fdiv_rn(y[2 * i + 1], s.scale));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Per-group FP8 of one pack of 8 rounded values y, in groups of `lanes` consecutive packs
// held by `lanes` consecutive lanes (aligned to `lanes`, which divides 32).  Every lane of
// the warp must call this (the group's amax is combined with shuffles); the pack's codes
// are returned, and the first lane of each group stores the group's scale when `store`.
__device__ __forceinline__ uint2 quant_pack_per_group(const float (&y)[8], int lanes, bool store, float* scale_slot) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(y[i]));
  for (int o = 1; o < lanes; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const Fp8Scale s = fp8_scale(a);
  if (store && (threadIdx.x & (unsigned)(lanes - 1)) == 0) st_f32(scale_slot, s.scale);
  return fp8_codes8(y, s);
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Warp maximum of values that are all >= 0 (magnitudes): their binary32 bit patterns order
// like the values, so one integer warp reduction gives the exact maximum in every lane.
__device__ __forceinline__ float warp_max_magnitude(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// Block-wide sum (MAX=false) or max of magnitudes (MAX=true, values >= 0) returned to every
// thread: a warp reduction, one barrier, then a reduction over the warp totals in every
// warp.  Both partners of a butterfly step combine the same two operands (and the integer
// maximum is exact), so every lane of every warp ends with the same bits.  `buf` holds one float per warp and must not be reused by
// another reduction before the next barrier.  When `any` is given, `flag` is OR-ed over the
// block in the same barrier and the result stored there (a caller agrees on a failure at
// no extra barrier).
template <bool MAX>
__device__ __forceinline__ float block_allreduce(float v, float* buf, bool flag = false, bool* any = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = MAX ? warp_max_magnitude(v) : warp_sum(v);
  if (lane == 0) buf[warp] = v;
  if (any != nullptr)
    *any = __syncthreads_or(flag) != 0;
  else
    __syncthreads();
  // identity of the sum, and of the max of magnitudes (every caller's values are >= 0)
  const float t = lane < nwarps ? buf[lane] : 0.0f;
  return MAX ? warp_max_magnitude(t) : warp_sum(t);
}

// ---------------------------------------------------------------------------
// thread-block clusters: one row split over csize CTAs, partial results exchanged
// through distributed shared memory (no multicast)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// Read a float from the shared memory of CTA `rank` of this cluster at the address that
// `local` has in this CTA.
__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Combine one value per CTA over the cluster (a sum, or the max of values >= 0); every
// thread of every CTA gets the same
// result.  `slot` is this CTA's published value (written by thread 0 before the call),
// `bcast` a one-float broadcast cell.  Starts with a full cluster barrier so every slot is
// written and visible.  The caller must not let a CTA exit while a peer may still read
// its slot: after the last exchange it executes cluster_arrive(), and cluster_wait()
// before returning.  Slots must not be rewritten between exchanges.
template <bool MAX>
__device__ __forceinline__ float cluster_gather(const float* slot, float* bcast, int csize) {
  cluster_sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float v = 0.0f;  // identity for the sum, and for the max of magnitudes
    if (lane < csize) v = ld_dsmem(slot, (uint32_t)lane);
    v = MAX ? warp_max_magnitude(v) : warp_sum(v);
    if (lane == 0) *bcast = v;
  }
  __syncthreads();
  return *bcast;
}

}  // namespace ar
