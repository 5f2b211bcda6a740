// Staged variant of the fused kernel: persistent CTAs, bulk asynchronous copies of whole
// rows (or, in the cluster form, of each CTA's slice of every row) into shared memory,
// S-deep pipeline.
//
// Same arithmetic as fused_kernel (ar_fused.cuh); only the data movement differs.  The
// grid holds as many CTAs as fit on the SMs at once (their shared-memory rings set the
// count); each loops over rows r = blockIdx.x + i * gridDim.x.  For each row one thread
// issues bulk global->shared copies (cp.async.bulk, the non-tensor form of TMA) of the N
// partial rows and the residual row into stage i % S and arms the stage's mbarrier with
// the byte count; while the CTA works on row i, rows i+1 .. i+S-1 are in flight (with
// S = 1, used when every row has its own CTA, the copy is the row's only one).  A stage is
// refilled as soon as the row's square-sum has been reduced (by then every thread has read
// its packs), so loads for later rows overlap the normalisation and the stores.  The
// weight packs a thread needs never change across rows and live in registers.
//
// Full tiles only (page "[HIP] [Perf] Specialize partial tiles in two-stage custom
// all-reduce", Proposed modifications: every thread executes the same number of
// barriers): the loop trip count is per CTA, identical for all its threads, and every
// barrier sits outside any per-thread predicate.
//
// Waits are bounded: a wait on a stage's mbarrier gives up after `wait_cycles` SM clock
// cycles, the CTA agrees on the failure in the row's square-sum barrier (an OR-reduction
// in the same barrier), records code 1 in `err`, waits (bounded again) for its own copies
// still in flight, and returns.
#pragma once

#include "ar_common.cuh"

namespace ar {

struct StagedParams {
  int stages;             // S, 1..4
  int row_bytes;          // h * 2
  int* err;               // device status word (0 = fine), written only on a timeout
  long long wait_cycles;  // bound of one mbarrier wait
  int stall_first;        // test hook: arm each CTA's first stage without issuing its copies, so
                          // that wait runs out (the failure path runs without any fault)
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Poll until the phase with `parity` completes or the cycle budget runs out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds_v4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// Address of `local` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
  return ra;
}

// Asynchronous stores into another CTA's shared memory that complete bytes on that CTA's
// mbarrier (both addresses from cluster_addr).
__device__ __forceinline__ void st_async_v2(uint32_t raddr, uint32_t a, uint32_t b, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
               "r"(a), "r"(b), "r"(rbar)
               : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t raddr, uint32_t v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr), "r"(v),
               "r"(rbar)
               : "memory");
}

// Poll an mbarrier whose phase other CTAs of the cluster complete (acquire at cluster scope,
// so their stores are visible after it) until the phase with `parity` completes or the cycle
// budget runs out.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > budget) return false;
  }
}

// The rows r = first + i * stride (i = 0, 1, ...) of one call, processed by this CTA
// through its shared-memory ring.  Shared by the persistent kernel and the batched one.
//
// Per row there are one or two block reductions: the square-sum, and with per-token FP8
// the amax of the rounded output.
//
// CL (cluster form, for rows longer than one CTA holds): the p.csize (2..8) CTAs of a cluster share
// each row, CTA rank r staging and processing packs [r * chunk, (r + 1) * chunk) of it
// (chunk = p.chunk_packs; the rows split exactly).  After each block reduction, thread 0
// sends the CTA's total to every peer with an asynchronous store into the peer's shared
// memory that completes on the peer's receive mbarrier (no cluster-wide barrier per row);
// every thread waits on its own CTA's receive barrier and adds the totals in rank order, so
// the whole cluster holds the same bits.  The failure flag of the bounded waits travels with
// the square-sum, so the CTAs of a cluster agree and leave together.  Receive buffers are
// double-buffered by row parity: a peer can only send row i + 2's total after this CTA sent
// row i + 1's, which it does after reading row i's.  Cluster barriers run only at the start
// (receive barriers initialised before any peer sends) and at the end (no CTA exits while a
// store to it may be in flight).
template <int DT, int N, int PPT, bool QUANT, bool CL = false>
__device__ __forceinline__ void staged_rows(const FusedParams& p, const StagedParams& sp, int64_t first,
                                            int64_t stride) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t full_bar[4];
  __shared__ float red_ss[2][32];
  __shared__ float red_amax[2][32];
  // cluster form: receive barriers [square-sum, amax][row parity] and buffers [parity][rank]
  __shared__ __align__(8) uint64_t rx_bar[2][2];
  __shared__ __align__(8) uint32_t rx_ss[2][8][2];  // {square-sum bits, failure flag}
  __shared__ __align__(8) uint32_t rx_am[2][8];

  const int csize = CL ? p.csize : 1;
  const int chunk = CL ? p.chunk_packs : p.row_packs;       // packs of a row this CTA handles
  const int col0 = CL ? (int)cluster_ctarank() * chunk : 0;  // first of them

  const int S = sp.stages;
  const bool has_res = p.res_in != nullptr;
  const int rows_per_stage = N + (has_res ? 1 : 0);
  const uint32_t row_bytes = (uint32_t)sp.row_bytes;
  const uint32_t stage_bytes = row_bytes * (uint32_t)rows_per_stage;
  const int64_t my_rows = first < p.m ? (p.m - first + stride - 1) / stride : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full_bar[s], 1);
    if (CL)
      for (int k = 0; k < 2; ++k)
        for (int b = 0; b < 2; ++b) mbar_init(&rx_bar[k][b], 1);
    mbar_fence_init();
  }
  // the first rows' inputs into L2 while the previous grid may still run (see prefetch_l2)
  if (p.prefetch && threadIdx.x == 0) {
    const int64_t pre = my_rows < S ? my_rows : S;
    for (int64_t i = 0; i < pre; ++i) {
      const size_t off = (size_t)(first + i * stride) * (size_t)(p.ld_in ? p.ld_in : (int64_t)p.h) * 2 +
                         (size_t)col0 * 16;
#pragma unroll
      for (int r = 0; r < N; ++r) prefetch_l2((const uint8_t*)p.x[r] + off, row_bytes);
      if (has_res) prefetch_l2((const uint8_t*)p.res_in + off, row_bytes);
    }
  }
  __syncthreads();
  if constexpr (CL) {  // every peer's receive barriers exist before anything is sent to them
    cluster_arrive();
    cluster_wait();
  }
  pdl_wait_and_release();

  auto issue = [&](int s, int64_t row) {
    uint8_t* dst = stage_mem + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
    if (sp.stall_first && row == first) return;  // nothing will complete this phase
    const size_t off = (size_t)row * (size_t)(p.ld_in ? p.ld_in : (int64_t)p.h) * 2 + (size_t)col0 * 16;
#pragma unroll
    for (int r = 0; r < N; ++r) bulk_g2s(dst + (size_t)r * row_bytes, (const uint8_t*)p.x[r] + off, row_bytes, &full_bar[s]);
    if (has_res) bulk_g2s(dst + (size_t)N * row_bytes, (const uint8_t*)p.res_in + off, row_bytes, &full_bar[s]);
  };

  if (threadIdx.x == 0) {
    const int64_t pre = my_rows < S ? my_rows : S;
    for (int64_t i = 0; i < pre; ++i) issue((int)i, first + i * stride);
  }

  // this thread's packs (fixed across rows) and their weight factors w' = w or 1 + w,
  // computed once: they are the same for every row
  bool valid[PPT];
  float wv[PPT][8];
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int pk = (int)threadIdx.x + k * (int)blockDim.x;
    valid[k] = pk < chunk;
    const int pkc = valid[k] ? pk : 0;
    if (p.skip_norm) {  // no norm: y = z * 1 * 1 = z exactly; the weight is not read
#pragma unroll
      for (int e = 0; e < 8; ++e) wv[k][e] = 1.0f;
    } else {
      unpack8<DT>(ld_keep(static_cast<const uint16_t*>(p.w) + (int64_t)(col0 + pkc) * 8), wv[k]);
      if (p.gemma) {
#pragma unroll
        for (int e = 0; e < 8; ++e) wv[k][e] = 1.0f + wv[k][e];
      }
    }
  }

  auto row_of = [&](int64_t i) { return first + i * stride; };
  auto out_base = [&](int64_t i) { return row_of(i) * (p.ld_out ? p.ld_out : (int64_t)p.h); };  // first output element
  auto pack_index = [&](int k) { return (int64_t)((int)threadIdx.x + k * (int)blockDim.x); };  // in the chunk
  auto gpack = [&](int k) { return (int64_t)col0 + pack_index(k); };                         // in the row

  // Wait for a row's stage s (bounded; `parity` selects the phase), then read it: rounded sum, residual add, this
  // thread's part of the square-sum.  A thread whose wait ran out still reads the stage
  // (in bounds; the values are discarded): the CTA agrees on the failure in the next barrier.
  auto read_row = [&](int s, uint32_t parity, uint4 (&z)[PPT], float (&zf)[PPT][8], float& ss) -> bool {
    const bool ok = mbar_wait_bounded(&full_bar[s], parity, sp.wait_cycles);
    const uint8_t* st = stage_mem + (size_t)s * stage_bytes;
    ss = 0.0f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      const int pkc = valid[k] ? (int)pack_index(k) : 0;
      // rank order: acc = x_0, then acc + x_1, ..., each an fp32 sum of an exact conversion
      float acc[8];
      unpack8<DT>(lds_v4(st + (size_t)pkc * 16), acc);
#pragma unroll
      for (int r = 1; r < N; ++r) add8<DT>(acc, lds_v4(st + (size_t)r * row_bytes + (size_t)pkc * 16));
      uint4 sv = pack8<DT>(acc);
      if (has_res) {  // z = round(res + s): the residual converted, the rounded sum added to it
        float rf[8];
        unpack8<DT>(lds_v4(st + (size_t)N * row_bytes + (size_t)pkc * 16), rf);
        add8<DT>(rf, sv);
        sv = pack8<DT>(rf);
      }
      z[k] = sv;
      unpack8<DT>(sv, zf[k]);
      if (valid[k]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(zf[k][e], zf[k][e], ss);
      }
    }
    return ok;
  };

  // After a failed wait on row i (stage s, phase parity): record the error and let this
  // CTA's own copies still in flight (rows i .. i+S-1) land before shared memory is released.
  auto fail_out = [&](int64_t i, int s, uint32_t parity) {
    if (threadIdx.x == 0) atomicExch(sp.err, 1);
    for (int64_t j = i; j < my_rows && j < i + S; ++j) {
      (void)mbar_wait_bounded(&full_bar[s], parity, sp.wait_cycles);
      if (++s == S) {
        s = 0;
        parity ^= 1u;
      }
    }
  };

  // Every thread has read row i's stage s: refill it with the row S iterations ahead.
  auto refill_after = [&](int64_t i, int s) {
    if (threadIdx.x == 0 && i + S < my_rows) {
      fence_proxy_async_smem();
      issue(s, row_of(i + S));
    }
  };

  // residual_out and the normalised row: stores z and y (16-bit or fp32); with FP8 leaves
  // the ROUNDED y in zf and returns this thread's part of its amax.
  auto normalise_row = [&](int64_t i, const uint4 (&z)[PPT], float (&zf)[PPT][8], float tot) -> float {
    const int64_t row_e = out_base(i);
    if (p.res_out != nullptr) {
#pragma unroll
      for (int k = 0; k < PPT; ++k)
        if (valid[k]) st_v4(static_cast<uint16_t*>(p.res_out) + row_e + gpack(k) * 8, z[k]);
    }
    const float inv = p.skip_norm ? 1.0f : rsqrtf(tot * p.inv_h + p.eps);
    uint4 y[PPT];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      float yf[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) yf[e] = (zf[k][e] * inv) * wv[k][e];
      y[k] = pack8<DT>(yf);
      if (p.out_f32 && valid[k]) {
        float* o = static_cast<float*>(p.out) + row_e + gpack(k) * 8;
        st_v4(o, make_uint4(__float_as_uint(yf[0]), __float_as_uint(yf[1]), __float_as_uint(yf[2]),
                            __float_as_uint(yf[3])));
        st_v4(o + 4, make_uint4(__float_as_uint(yf[4]), __float_as_uint(yf[5]), __float_as_uint(yf[6]),
                                __float_as_uint(yf[7])));
      }
      if (QUANT) {
        unpack8<DT>(y[k], zf[k]);  // zf now holds the ROUNDED output y
        if (valid[k]) {
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(zf[k][e]));
        }
      }
    }
    if (p.out != nullptr && !p.out_f32) {
#pragma unroll
      for (int k = 0; k < PPT; ++k)
        if (valid[k]) st_v4(static_cast<uint16_t*>(p.out) + row_e + gpack(k) * 8, y[k]);
    }
    return amax;
  };

  // Per-token FP8 codes of row i from its rounded y and the row's amax.
  auto quantise_row = [&](int64_t i, const float (&yq)[PPT][8], float am) {
    const int64_t row_e = out_base(i);
    const Fp8Scale fs = fp8_scale(am);  // an all-zero row keeps codes 0 (no division)
    if (threadIdx.x == 0 && col0 == 0) st_f32(p.scale + row_of(i), fs.scale);  // one CTA of a cluster
#pragma unroll
    for (int k = 0; k < PPT; ++k)
      if (valid[k]) st_v2(p.q + row_e + gpack(k) * 8, fp8_codes8(yq[k], fs));
  };

  // Cluster form: combine this CTA's square-sum (and failure flag) or amax of row i with the
  // other CTAs' (see the comment above the function); no-ops without a cluster.
  const uint32_t me = CL ? cluster_ctarank() : 0;
  auto cluster_sum = [&](int64_t i, float& tot, bool& failed) {
    if constexpr (CL) {
      const int b = (int)(i & 1);
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&rx_bar[0][b], (uint32_t)(csize - 1) * 8u);
        for (int r = 0; r < csize; ++r)
          if (r != (int)me)
            st_async_v2(cluster_addr(&rx_ss[b][me][0], (uint32_t)r), __float_as_uint(tot), failed ? 1u : 0u,
                        cluster_addr(&rx_bar[0][b], (uint32_t)r));
      }
      const bool ok = mbar_wait_cluster_bounded(&rx_bar[0][b], (uint32_t)((i >> 1) & 1), 4 * sp.wait_cycles);
      float t = 0.0f;
      bool f = failed || !ok;
      for (int r = 0; r < csize; ++r) {
        if (r == (int)me) {
          t += tot;
        } else {
          t += __uint_as_float(rx_ss[b][r][0]);
          f = f || rx_ss[b][r][1] != 0u;
        }
      }
      tot = t;
      failed = f;
    }
  };
  auto cluster_max = [&](int64_t i, float am) -> float {
    if constexpr (CL) {
      const int b = (int)(i & 1);
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&rx_bar[1][b], (uint32_t)(csize - 1) * 4u);
        for (int r = 0; r < csize; ++r)
          if (r != (int)me)
            st_async_b32(cluster_addr(&rx_am[b][me], (uint32_t)r), __float_as_uint(am),
                         cluster_addr(&rx_bar[1][b], (uint32_t)r));
      }
      const bool ok = mbar_wait_cluster_bounded(&rx_bar[1][b], (uint32_t)((i >> 1) & 1), 4 * sp.wait_cycles);
      if (!ok && threadIdx.x == 0) atomicExch(sp.err, 1);
      float a = 0.0f;
      for (int r = 0; r < csize; ++r) a = fmaxf(a, r == (int)me ? am : __uint_as_float(rx_am[b][r]));
      return a;
    } else {
      return am;
    }
  };
  // no CTA of a cluster leaves while a store to it may still be in flight
  auto cluster_leave = [&]() {
    if constexpr (CL) {
      cluster_arrive();
      cluster_wait();
    }
  };

  // stage and phase of row i, kept incrementally (i % S and i / S would be 64-bit divisions)
  int s = 0;
  uint32_t parity = 0;
  for (int64_t i = 0; i < my_rows; ++i) {
    uint4 z[PPT];
    float zf[PPT][8], ss;
    const bool ok = read_row(s, parity, z, zf, ss);
    float tot = 0.0f;
    bool failed;
    if (!p.skip_norm)
      tot = block_allreduce<false>(ss, red_ss[i & 1], !ok, &failed);
    else
      failed = __syncthreads_or(!ok) != 0;
    cluster_sum(i, tot, failed);
    if (failed) {
      fail_out(i, s, parity);
      cluster_leave();
      return;
    }
    refill_after(i, s);
    const float amax = normalise_row(i, z, zf, tot);
    if constexpr (QUANT) {
      if (p.group_lanes) {  // per group: lanes of a group combine, no block reduction
        const int64_t row_e = out_base(i);
#pragma unroll
        for (int k = 0; k < PPT; ++k) {
          const int pk = col0 + (int)threadIdx.x + k * (int)blockDim.x;
          const uint2 cw = quant_pack_per_group(zf[k], p.group_lanes, valid[k],
                                                p.scale + row_of(i) * (int64_t)p.ngroups + pk / p.group_lanes);
          if (valid[k]) st_v2(p.q + row_e + (int64_t)pk * 8, cw);
        }
      } else {  // per token: the row's amax over the block
        quantise_row(i, zf, cluster_max(i, block_allreduce<true>(amax, red_amax[i & 1])));
      }
    }
    if (++s == S) {
      s = 0;
      parity ^= 1u;
    }
  }
  cluster_leave();
}

// The explicit minimum of one CTA per SM for 1 and 2 packs per thread lets ptxas give each
// thread more registers (about 80 instead of 55-60 at 2 packs) and keep more shared-memory
// loads in flight; measured faster in every one-CTA-per-SM configuration.
template <int DT, int N, int PPT, bool QUANT>
__global__ void __launch_bounds__(1024 / PPT, (PPT <= 2 ? 1 : 0)) fused_staged_kernel(const FusedParams p, const StagedParams sp) {
  staged_rows<DT, N, PPT, QUANT>(p, sp, blockIdx.x, gridDim.x);
}

// Cluster form for rows longer than one CTA holds (p.csize CTAs per row, each p.chunk_packs
// packs, PPT per thread); the grid is a whole number of clusters, each looping over rows
// r = cluster index + i * clusters.
template <int DT, int N, int PPT, bool QUANT>
__global__ void __launch_bounds__(1024 / PPT, 1) fused_staged_cluster_kernel(const FusedParams p, const StagedParams sp) {
  staged_rows<DT, N, PPT, QUANT, true>(p, sp, blockIdx.x / p.csize, gridDim.x / p.csize);
}

// ---------------------------------------------------------------------------
// Batched form: up to kMaxBatch independent calls (same N, element type and options) in
// one launch.  CTA b serves row b - row_start[c] of the call c with
// row_start[c] <= b < row_start[c + 1], one row per CTA, with one shared-memory stage.
// ---------------------------------------------------------------------------
constexpr int kMaxBatch = 16;

struct BatchParams {
  int count;
  int64_t row_start[kMaxBatch + 1];
  StagedParams sp;  // row_bytes is per call: taken from call[c].h
  FusedParams call[kMaxBatch];
};

template <int DT, int N, int PPT, bool QUANT>
__global__ void __launch_bounds__(1024 / PPT, (PPT <= 2 ? 1 : 0)) fused_batch_kernel(const BatchParams bp) {
  int c = 0;
  while (c + 1 < bp.count && (int64_t)blockIdx.x >= bp.row_start[c + 1]) ++c;
  const int64_t row = (int64_t)blockIdx.x - bp.row_start[c];
  StagedParams sp = bp.sp;
  sp.row_bytes = bp.call[c].h * 2;
  staged_rows<DT, N, PPT, QUANT>(bp.call[c], sp, row, bp.call[c].m);
}

}  // namespace ar
