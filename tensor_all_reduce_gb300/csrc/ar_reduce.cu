// Plain N-way sum-reduce: out = round_T(sum_r (float)x_r), fp32 accumulation in rank
// order 0..N-1, one rounding (page "[OUTDATED] perf: optimize fused AllReduce + RMSNorm
// (custom_all_reduce)", Technical Details / 2stage, flat reduce-scatter: one thread per
// 16-byte pack across all inputs, no shared memory, no block barrier).
//
// Tiling follows page "[HIP] [Perf] Specialize partial tiles in two-stage custom
// all-reduce", Proposed modifications: the main loop runs over complete tiles only
// (blockDim * UNROLL packs, no predicates); with HAS_TAIL the leftover packs and the
// leftover elements (numel not a multiple of the pack) are reduced by the block that would
// own the next tile, each by its original owner thread index.  Aligned sizes use
// HAS_TAIL = false and carry no tail code at all.  The kernels contain no barrier.
#include "ar_common.cuh"
#include "ar_launch.h"

namespace ar {

template <int DT>
struct PackT;

template <>
struct PackT<kF32> {
  static constexpr int kElems = 4;
  __device__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ static float load1(const void* b, int64_t i) { return ld_f32(static_cast<const float*>(b) + i); }
  __device__ static void store1(void* b, int64_t i, float v) { st_f32(static_cast<float*>(b) + i, v); }
};

template <int DT>
struct PackT16 {
  static constexpr int kElems = 8;
  __device__ static void unpack(const uint4& v, float (&f)[8]) { unpack8<DT>(v, f); }
  __device__ static uint4 pack(const float (&f)[8]) { return pack8<DT>(f); }
  __device__ static float load1(const void* b, int64_t i) {
    return to_f32<DT>(ld_u16(static_cast<const uint16_t*>(b) + i));
  }
  __device__ static void store1(void* b, int64_t i, float v) {
    st_u16(static_cast<uint16_t*>(b) + i, round1<DT>(v));
  }
};
template <>
struct PackT<kF16> : PackT16<kF16> {};
template <>
struct PackT<kBF16> : PackT16<kBF16> {};

template <int DT, int N>
__device__ __forceinline__ uint4 reduce_one_pack(const ReduceParams& p, int64_t pk) {
  using P = PackT<DT>;
  constexpr int E = P::kElems;
  float acc[E];
  P::unpack(ld_stream(static_cast<const uint4*>(p.x[0]) + pk), acc);
#pragma unroll
  for (int r = 1; r < N; ++r) {
    float t[E];
    P::unpack(ld_stream(static_cast<const uint4*>(p.x[r]) + pk), t);
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = acc[i] + t[i];
  }
  return P::pack(acc);
}

template <int DT, int N>
__device__ __forceinline__ void reduce_one_elem(const ReduceParams& p, int64_t e) {
  using P = PackT<DT>;
  float acc = P::load1(p.x[0], e);
#pragma unroll
  for (int r = 1; r < N; ++r) acc = acc + P::load1(p.x[r], e);
  P::store1(p.out, e, acc);
}

template <int DT, int N, int UNROLL, bool HAS_TAIL>
__global__ void __launch_bounds__(256) reduce_vec_kernel(const ReduceParams p) {
  const int64_t bs = blockDim.x;
  const int64_t tile = bs * UNROLL;
  // this block's first tile (or the tail packs it owns) into L2 while the previous grid may
  // still run (see prefetch_l2)
  if (p.prefetch && threadIdx.x == 0) {
    int64_t first = -1, packs = 0;
    if ((int64_t)blockIdx.x < p.full_tiles) {
      first = (int64_t)blockIdx.x * tile;
      packs = tile;
    } else if (HAS_TAIL && blockIdx.x == (unsigned)(p.full_tiles % gridDim.x)) {
      first = p.full_tiles * tile;
      packs = p.npacks - first;
    }
    if (packs > 0) {
#pragma unroll
      for (int r = 0; r < N; ++r) prefetch_l2(static_cast<const uint4*>(p.x[r]) + first, (uint32_t)(packs * 16));
    }
  }
  pdl_wait_and_release();
  uint4* out = static_cast<uint4*>(p.out);
  for (int64_t t = blockIdx.x; t < p.full_tiles; t += gridDim.x) {
    const int64_t base = t * tile + threadIdx.x;
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = reduce_one_pack<DT, N>(p, base + u * bs);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) st_v4(out + base + u * bs, v[u]);
  }
  if constexpr (HAS_TAIL) {
    if (blockIdx.x == (unsigned)(p.full_tiles % gridDim.x)) {
      const int64_t base = p.full_tiles * tile + threadIdx.x;
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int64_t pk = base + u * bs;
        if (pk < p.npacks) st_v4(out + pk, reduce_one_pack<DT, N>(p, pk));
      }
      const int64_t e = p.npacks * PackT<DT>::kElems + threadIdx.x;
      if (e < p.numel) reduce_one_elem<DT, N>(p, e);
    }
  }
}

// Element-wise form for pointers that are not 16-byte aligned.
template <int DT, int N>
__global__ void __launch_bounds__(256) reduce_scalar_kernel(const ReduceParams p) {
  pdl_wait_and_release();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.numel; e += stride)
    reduce_one_elem<DT, N>(p, e);
}

// ---------------------------------------------------------------------------
// host-side selection of the instantiation
// ---------------------------------------------------------------------------

template <int DT, int N>
static const void* pick_reduce_n(int unroll, bool vec, bool has_tail) {
  if (!vec) return (const void*)&reduce_scalar_kernel<DT, N>;
  if (unroll == 1)
    return has_tail ? (const void*)&reduce_vec_kernel<DT, N, 1, true>
                    : (const void*)&reduce_vec_kernel<DT, N, 1, false>;
  return has_tail ? (const void*)&reduce_vec_kernel<DT, N, 4, true>
                  : (const void*)&reduce_vec_kernel<DT, N, 4, false>;
}

template <int DT>
static const void* pick_reduce_dt(int n, int unroll, bool vec, bool has_tail) {
  switch (n) {
    case 1: return pick_reduce_n<DT, 1>(unroll, vec, has_tail);
    case 2: return pick_reduce_n<DT, 2>(unroll, vec, has_tail);
    case 3: return pick_reduce_n<DT, 3>(unroll, vec, has_tail);
    case 4: return pick_reduce_n<DT, 4>(unroll, vec, has_tail);
    case 5: return pick_reduce_n<DT, 5>(unroll, vec, has_tail);
    case 6: return pick_reduce_n<DT, 6>(unroll, vec, has_tail);
    case 7: return pick_reduce_n<DT, 7>(unroll, vec, has_tail);
    case 8: return pick_reduce_n<DT, 8>(unroll, vec, has_tail);
    default: return nullptr;
  }
}

const void* reduce_kernel(int dtype, int n, int unroll, bool vec, bool has_tail) {
  switch (dtype) {
    case kF32: return pick_reduce_dt<kF32>(n, unroll, vec, has_tail);
    case kF16: return pick_reduce_dt<kF16>(n, unroll, vec, has_tail);
    case kBF16: return pick_reduce_dt<kBF16>(n, unroll, vec, has_tail);
    default: return nullptr;
  }
}

}  // namespace ar
