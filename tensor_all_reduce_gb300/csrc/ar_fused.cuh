// Fused N-way reduce + residual add + RMSNorm (+ per-token FP8 E4M3) kernel.
//
// Semantics (page "[HIP] fix(custom-ar): gfx1250 fused all-reduce + RMSNorm", Changes):
// ranks are summed in fixed order in fp32 and rounded once to the storage type, the
// residual is added and rounded again exactly as the unfused rmsnorm2d_fwd_with_add
// does, the row is normalised (plain or gemma (1 + w) weight), and the optional FP8
// epilogue quantises the ROUNDED output per row with the steps of
// dynamic_per_token_scaled_quant, writing the 16-bit mirror as well.
//
// Work decomposition (GB300 design, not the pages'): a row of h elements is split over a
// thread-block cluster of `csize` CTAs (csize = 1: one CTA per row).  Each CTA owns a
// contiguous chunk of 16-byte packs; each thread owns PPT packs strided by blockDim.
// The row's square-sum and, with FP8, its amax are combined warp -> block (shared
// memory) -> cluster (distributed shared memory).  Small-M decode shapes use csize > 1 so
// that the few rows still spread over many SMs; large M uses csize = 1.  On device memory the
// staged kernel (ar_staged.cuh) takes every 16-byte-aligned row of up to 8192 elements; this
// kernel serves buffers in host memory, rows that are not 16-byte aligned (VEC = false) and
// rows longer than the staged cluster form takes, and runs when forced.
//
// VEC = true : every pack is a full, 16-byte-aligned group of 8 elements (h % 8 == 0 and
//              all row starts aligned); one 128-bit load per pack and partial.
// VEC = false: the tail specialisation for rows whose length is not a multiple of the
//              pack or whose pointers are not 16-byte aligned: the same packs of 8
//              elements, loaded element by element with a per-element predicate
//              (page "[HIP] [Perf] Specialize partial tiles in two-stage custom
//              all-reduce", Proposed modifications: leftover elements take a predicated
//              path; no barrier ever sits inside a loop whose trip count differs
//              between threads).
#pragma once

#include "ar_common.cuh"

namespace ar {

// Load one pack (8 elements starting at element index e0 of `base`) as floats.
// Elements at or beyond `limit` (scalar variant only) read as 0.
template <int DT, bool VEC, bool STREAM>
__device__ __forceinline__ void load_pack(const void* base, int64_t e0, int64_t limit, float (&f)[8]) {
  const uint16_t* b = static_cast<const uint16_t*>(base);
  if constexpr (VEC) {
    uint4 v = STREAM ? ld_stream(b + e0) : ld_keep(b + e0);
    unpack8<DT>(v, f);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = (e0 + i < limit) ? to_f32<DT>(ld_u16(b + e0 + i)) : 0.0f;
  }
}

// acc[i] = acc[i] + x_i for the pack at base[e0 .. e0 + 8) (in the element-wise form,
// elements at or beyond `limit` count as 0): each sum is one fp32 rounding of an exact
// conversion, as mixed-precision adds in the vector form.
template <int DT, bool VEC, bool STREAM>
__device__ __forceinline__ void load_add_pack(const void* base, int64_t e0, int64_t limit, float (&acc)[8]) {
  const uint16_t* b = static_cast<const uint16_t*>(base);
  if constexpr (VEC) {
    add8<DT>(acc, STREAM ? ld_stream(b + e0) : ld_keep(b + e0));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc[i] + ((e0 + i < limit) ? to_f32<DT>(ld_u16(b + e0 + i)) : 0.0f);
  }
}

// Store one pack of 16-bit values (already rounded, packed in a uint4).
template <bool VEC>
__device__ __forceinline__ void store_pack(void* base, int64_t e0, int64_t limit, const uint4& v) {
  uint16_t* b = static_cast<uint16_t*>(base);
  if constexpr (VEC) {
    st_v4(b + e0, v);
  } else {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (e0 + i < limit) st_u16(b + e0 + i, (uint16_t)((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu));
  }
}

// Store eight fp32 values (elements e0 .. e0+7 of an fp32 [m, h] array).
template <bool VEC>
__device__ __forceinline__ void store_f32x8(void* base, int64_t e0, int64_t limit, const float (&f)[8]) {
  float* b = static_cast<float*>(base);
  if constexpr (VEC) {
    st_v4(b + e0, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                             __float_as_uint(f[3])));
    st_v4(b + e0 + 4, make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                                 __float_as_uint(f[7])));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (e0 + i < limit) st_f32(b + e0 + i, f[i]);
  }
}

template <int DT, int N, int PPT, bool QUANT, bool VEC>
__global__ void __launch_bounds__(1024 / PPT) fused_kernel(const FusedParams p) {
  __shared__ float red_ss[32];
  __shared__ float red_amax[32];
  __shared__ float slot_ss, slot_amax, bcast;

  const int csize = p.csize;
  const int crank = (int)(blockIdx.x % (unsigned)csize);  // == %cluster_ctarank for (csize,1,1) clusters
  const int64_t row = blockIdx.x / (unsigned)csize;
  const int pk_begin = crank * p.chunk_packs;
  const int pk_end = min(pk_begin + p.chunk_packs, p.row_packs);
  // rows may be padded: inputs and outputs have their own row strides (0 means h)
  const int64_t row_i = row * (p.ld_in ? p.ld_in : (int64_t)p.h);     // first input element of the row
  const int64_t row_i_end = row_i + p.h;
  const int64_t row_e = row * (p.ld_out ? p.ld_out : (int64_t)p.h);   // first output element of the row
  const int64_t row_end = row_e + p.h;         // one past the row's last output element

  // this CTA's slice of the row into L2 while the previous grid may still run (see prefetch_l2)
  if constexpr (VEC) {
    if (p.prefetch && threadIdx.x == 0 && pk_end > pk_begin) {
      const uint32_t bytes = (uint32_t)(pk_end - pk_begin) * 16u;
      const int64_t e0 = row_i + (int64_t)pk_begin * 8;
#pragma unroll
      for (int r = 0; r < N; ++r) prefetch_l2(static_cast<const uint16_t*>(p.x[r]) + e0, bytes);
      if (p.res_in != nullptr) prefetch_l2(static_cast<const uint16_t*>(p.res_in) + e0, bytes);
    }
  }
  pdl_wait_and_release();

  // ---- phase 1: loads of every pack this thread owns, then the reduction --------------
  // Indices of packs beyond the chunk are clamped to the chunk's first pack so that all
  // loads are unconditional and can be issued back to back; their results are discarded.
  uint4 z[PPT];
  uint4 wpk[PPT];
  bool valid[PPT];
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int pk = pk_begin + (int)threadIdx.x + k * (int)blockDim.x;
    valid[k] = pk < pk_end;
    const int pkc = valid[k] ? pk : pk_begin;
    const int64_t e0 = row_i + (int64_t)pkc * 8;
    const int64_t lim = valid[k] ? row_i_end : row_i;  // scalar variant: nothing for clamped packs
    float acc[8];
    load_pack<DT, VEC, true>(p.x[0], e0, lim, acc);
#pragma unroll
    for (int r = 1; r < N; ++r) load_add_pack<DT, VEC, true>(p.x[r], e0, lim, acc);  // fp32, rank order
    uint4 s = pack8<DT>(acc);                              // one rounding to T
    if (p.res_in != nullptr) {                             // z = round(res + s)
      float rf[8];
      load_pack<DT, VEC, true>(p.res_in, e0, lim, rf);
      add8<DT>(rf, s);
      s = pack8<DT>(rf);                                   // second rounding to T
    }
    z[k] = s;
    // weight row: 8 consecutive entries starting at column pkc * 8 (none without the norm)
    if (!p.skip_norm) {
      float wf[8];
      const int64_t c0 = (int64_t)pkc * 8;
      load_pack<DT, VEC, false>(p.w, c0, valid[k] ? (int64_t)p.h : 0, wf);
      wpk[k] = pack8<DT>(wf);                              // exact: wf are T values
    } else {
      wpk[k] = make_uint4(0, 0, 0, 0);
    }
    if (valid[k]) {
      float zf[8];
      unpack8<DT>(z[k], zf);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(zf[i], zf[i], ss);  // absent elements are 0
    }
  }
  if (p.res_out != nullptr) {
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      if (valid[k]) {
        const int pk = pk_begin + (int)threadIdx.x + k * (int)blockDim.x;
        store_pack<VEC>(p.res_out, row_e + (int64_t)pk * 8, row_end, z[k]);
      }
    }
  }

  // ---- row square-sum: warp -> block -> cluster ------------------------------------
  float inv = 1.0f;  // without the norm y = z * 1 * 1 = z exactly
  if (!p.skip_norm) {
    float tot = block_allreduce<false>(ss, red_ss);
    if (csize > 1) {
      if (threadIdx.x == 0) slot_ss = tot;
      tot = cluster_gather<false>(&slot_ss, &bcast, csize);
    }
    inv = rsqrtf(tot * p.inv_h + p.eps);
  }

  // ---- phase 2: normalise, weight, round ---------------------------------------------
  uint4 y[PPT];
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    float zf[8], wf[8], yf[8];
    unpack8<DT>(z[k], zf);
    unpack8<DT>(wpk[k], wf);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float wv = p.skip_norm ? 1.0f : (p.gemma ? 1.0f + wf[i] : wf[i]);
      yf[i] = (zf[i] * inv) * wv;
    }
    y[k] = pack8<DT>(yf);
    if (p.out_f32 && valid[k]) {
      const int pk = pk_begin + (int)threadIdx.x + k * (int)blockDim.x;
      store_f32x8<VEC>(p.out, row_e + (int64_t)pk * 8, row_end, yf);
    }
    if (QUANT && valid[k]) {
      float yr[8];
      unpack8<DT>(y[k], yr);                               // amax of the ROUNDED output
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(yr[i]));
    }
  }
  if (p.out != nullptr && !p.out_f32) {
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      if (valid[k]) {
        const int pk = pk_begin + (int)threadIdx.x + k * (int)blockDim.x;
        store_pack<VEC>(p.out, row_e + (int64_t)pk * 8, row_end, y[k]);
      }
    }
  }

  // ---- FP8 epilogue ----------------------------------------------------------------
  if (QUANT && p.group_lanes) {  // per group: no block reduction, lanes of a group combine
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      const int pk = pk_begin + (int)threadIdx.x + k * (int)blockDim.x;
      float yr[8];
      unpack8<DT>(y[k], yr);
      const uint2 cw = quant_pack_per_group(yr, p.group_lanes, valid[k],
                                            p.scale + row * (int64_t)p.ngroups + pk / p.group_lanes);
      if (!valid[k]) continue;
      const int64_t e0 = row_e + (int64_t)pk * 8;
      if constexpr (VEC) {
        st_v2(p.q + e0, cw);
      } else {
        const uint32_t c2[2] = {cw.x, cw.y};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (e0 + i < row_end) st_u8(p.q + e0 + i, (uint8_t)((c2[i >> 2] >> (8 * (i & 3))) & 0xFFu));
      }
    }
  } else if constexpr (QUANT) {
    float am = block_allreduce<true>(amax, red_amax);
    if (csize > 1) {
      if (threadIdx.x == 0) slot_amax = am;
      am = cluster_gather<true>(&slot_amax, &bcast, csize);
    }
    const Fp8Scale fs = fp8_scale(am);  // an all-zero row has scale 0 and all codes 0
    if (crank == 0 && threadIdx.x == 0) st_f32(p.scale + row, fs.scale);
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      if (!valid[k]) continue;
      const int pk = pk_begin + (int)threadIdx.x + k * (int)blockDim.x;
      float yr[8];
      unpack8<DT>(y[k], yr);
      const uint2 cw = fp8_codes8(yr, fs);
      const int64_t e0 = row_e + (int64_t)pk * 8;
      if constexpr (VEC) {
        st_v2(p.q + e0, cw);
      } else {
        const uint32_t c2[2] = {cw.x, cw.y};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (e0 + i < row_end) st_u8(p.q + e0 + i, (uint8_t)((c2[i >> 2] >> (8 * (i & 3))) & 0xFFu));
      }
    }
  }

  if (csize > 1) {
    cluster_arrive();  // done reading peers' slots
    cluster_wait();    // and no peer still reads ours
  }
}

}  // namespace ar
