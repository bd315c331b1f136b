// Device-side helpers shared by the librkv kernels (sm_103a).
//
// Small wrappers around PTX: bf16 unpacking, the m16n8k16 bf16 tensor-core MMA,
// ldmatrix, cp.async, mbarrier waits with a time limit, and bulk (TMA engine)
// global->shared copies.  Nothing here is specific to one kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rkv.h"

namespace rkv {

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ float bf16_f(uint16_t x) { return __uint_as_float(uint32_t(x) << 16); }

// Two floats -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ tensor core
// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate (row.col).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// ------------------------------------------------------------------ cp.async (16 B)
// src_bytes = 0 writes 16 zero bytes without reading global memory.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}

// Time limit of every wait on an mbarrier in the library's kernels: far beyond any
// copy's latency, short enough that a wait nothing will end returns control.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Wait for phase `parity` of `bar` for at most limit_ns; false when the time ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_ns() - t0 > limit_ns) return false;
  }
}

// Bulk copy (TMA engine) of `bytes` (multiple of 16, 16-B aligned ends) from global to
// this CTA's shared memory; completion is signalled on `bar` as transaction bytes.
// A hint: fetch [src, src + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
// Nothing waits for it, and L2 never serves stale data, so it may run before the
// writes it would otherwise have to follow.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

// The same for the one 128-byte line holding `p` (any alignment).
__device__ __forceinline__ void prefetch_line_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p)); }

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}


// Tiled TMA load of one box of a 2-D tensor map into this CTA's shared memory;
// completion is signalled on `bar` as transaction bytes.  `map` must live in
// parameter, constant or global memory (a __grid_constant__ kernel parameter).
// The innermost coordinate x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 2^x by the special function unit's single instruction (PTX ex2.approx.ftz.f32):
// relative error of a few ulps, results below 2^-126 flushed to zero.  Used where the
// exponential is the inner loop's cost (the scoring epilogues, the attention's online
// softmax) and in the merges of partial softmax states.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch (PTX griddepcontrol): wait until the prerequisite grid
// on the stream has completed and its memory writes are visible (a no-op when the
// kernel was not launched as a dependent), and allow the dependent grid to be
// scheduled.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Dynamic shared memory rounded up to a 1024-byte boundary (the 128-byte swizzle atom).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// ------------------------------------------------------------------ tcgen05 (5th-gen tensor cores)
// Tensor memory (TMEM): 128 lanes x 512 columns of 32-bit cells per SM.  Addresses are
// (lane << 16) | column.  One warp allocates and frees; the base lands in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 in, fp32 accumulate; issued by one thread.
// adesc / bdesc: shared-memory matrix descriptors; idesc: instruction descriptor.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 consecutive columns of this thread's TMEM lane (the warp covers 32 lanes), with
// the wait for the load in the same statement so no use of r can move above it.
__device__ __forceinline__ void tc_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 operand stored as TMA writes it with
// 128-byte swizzle: rows of 128 B (64 elements of K), 8-row groups 1024 B apart, the
// atom 1024-byte aligned.  Fields: start address >> 4 (bits 0-13), leading byte offset
// >> 4 (16-29, unused by swizzled K-major layouts), stride byte offset >> 4 (32-45),
// the fixed 0b001 of bits 46-48, swizzle mode 2 = 128 B (61-63).  A K step of 16
// elements inside the 128-B row is a +32 B start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both K-major:
// D format (bits 4-5) = 1 (f32), A format (7-9) = 1 (bf16), B format (10-12) = 1 (bf16),
// N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ errors
__device__ __forceinline__ void flag_error(int32_t* word, int32_t bit) {
  if (word) atomicOr(word, bit);
}

// ------------------------------------------------------------------ adaptive-bin top-k
// Top k of n uint32 keys, ordered by (key descending, index ascending), for
// 1 <= k < n: the ascending indices go to out[0..k) (and out2, when not null).
//
// The key interval [lo, hi] that holds the k-th key shrinks by histograms of 1024
// bins laid linearly over it (the first over [min key, max key]); a round ends with
// the bin holding the k-th key.  Once that bin holds at most kTkCand keys, the
// boundary key and index (T, t) come from ranking the bin's keys among themselves,
// and the selection is {key > hi} + {key in [lo, hi] with (key, -index) >= (T, -t)}.
// If the interval has shrunk to a single key value with more keys than that, the
// equal keys are taken by ascending index.  Keys are order-preserving images of
// floats in practice, so one round usually leaves a handful of candidates.
//
// Thread t owns the contiguous keys [t seg, t seg + seg), seg odd: strided
// shared-memory reads then hit distinct banks, a run of equal keys adds to the
// histogram once, and the compaction is one pass with one block scan.  `key(i)` is
// called several times for each i in [0, n); every thread of the block calls this.
constexpr int kTkBins = 1024;
constexpr int kTkCand = 32;
constexpr int kTkCandFlat = 64;  // the candidate cap of topk_flat (two ranking warps)
template <int NT, int NBINS = kTkBins>
struct TopkSmem {
  alignas(16) uint32_t hist[NBINS];
  alignas(16) int cand[kTkCandFlat];
  alignas(16) uint32_t ckey[kTkCandFlat];
  uint32_t wlo[NT / 32], whi[NT / 32];
  int wa[NT / 32], wb[NT / 32];
  int ncand, bstar, need, nb, tidx;
  uint32_t tkey;
};

// take(pos, i) receives every selected index i with its position pos in the ascending
// list (each from exactly one thread).
template <int NT, class KeyFn, class TakeFn>
__device__ void topk_adaptive_fn(int n, int k, KeyFn key, TopkSmem<NT>& ts, TakeFn take) {
  static_assert(NT % 32 == 0 && kTkBins % NT == 0, "bins must split evenly over the threads");
  constexpr int NW = NT / 32;
  constexpr int BPT = kTkBins / NT;  // bins per thread
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = ((n + NT - 1) / NT) | 1;
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);

  // 1. the key range
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll 4
  for (int i = s0; i < s1; ++i) {
    const uint32_t u = key(i);
    lo = min(lo, u);
    hi = max(hi, u);
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    ts.wlo[warp] = lo;
    ts.whi[warp] = hi;
  }
  if (tid == 0) ts.ncand = 0;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    lo = min(lo, ts.wlo[w]);
    hi = max(hi, ts.whi[w]);
  }

  // 2. shrink [lo, hi]; `need` of the `nin` keys inside it are taken
  int need = k, nin = n;
  while (nin > kTkCand && lo != hi) {
    const uint32_t range = hi - lo;
    const int shift = range < (uint32_t)kTkBins ? 0 : (32 - __clz(range)) - 10;  // (range >> shift) < 1024
    for (int i = tid; i < kTkBins; i += NT) ts.hist[i] = 0u;
    __syncthreads();
    int run_bin = -1, run = 0;
#pragma unroll 4
    for (int i = s0; i < s1; ++i) {
      const uint32_t u = key(i);
      const int bin = (u >= lo && u <= hi) ? (int)((u - lo) >> shift) : -1;
      if (bin != run_bin) {
        if (run_bin >= 0) atomicAdd(&ts.hist[run_bin], (uint32_t)run);
        run_bin = bin;
        run = 0;
      }
      ++run;
    }
    if (run_bin >= 0) atomicAdd(&ts.hist[run_bin], (uint32_t)run);
    __syncthreads();
    uint32_t c[BPT];
    if constexpr (BPT % 4 == 0) {
#pragma unroll
      for (int j = 0; j < BPT; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(&ts.hist[tid * BPT + j]);
        c[j] = v.x;
        c[j + 1] = v.y;
        c[j + 2] = v.z;
        c[j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < BPT; ++j) c[j] = ts.hist[tid * BPT + j];
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) s += (int)c[j];
    int incl = s;  // sum over the lanes >= this one
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += y;
    }
    if (lane == 0) ts.wa[warp] = incl;
    __syncthreads();
    int above = incl - s;  // keys in the bins above this thread's
    for (int w = warp + 1; w < NW; ++w) above += ts.wa[w];
    if (above < need && above + s >= need) {
      int acc = above;
#pragma unroll
      for (int j = BPT - 1; j >= 0; --j) {
        if (acc + (int)c[j] >= need) {
          ts.bstar = tid * BPT + j;
          ts.need = need - acc;
          ts.nb = (int)c[j];
          break;
        }
        acc += (int)c[j];
      }
    }
    __syncthreads();
    const uint32_t nlo = lo + ((uint32_t)ts.bstar << shift);
    hi = shift == 0 ? nlo : min(hi, nlo + ((1u << shift) - 1u));
    lo = nlo;
    need = ts.need;
    nin = ts.nb;
    // the next round's first barrier orders these reads before the next writes
  }

  // 3. the boundary pair (T, t) among at most kTkCand candidates
  const bool all_in = need == nin;                // every key in [lo, hi] is taken
  const bool by_index = !all_in && nin > kTkCand;  // then lo == hi
  if (!by_index && !all_in) {
    for (int i = s0; i < s1; ++i) {
      const uint32_t u = key(i);
      if (u >= lo && u <= hi) {
        const int slot = atomicAdd(&ts.ncand, 1);
        if (slot < kTkCand) {
          ts.cand[slot] = i;
          ts.ckey[slot] = u;
        }
      }
    }
    __syncthreads();
    const int nc = min(ts.ncand, kTkCand);
    for (int j = tid; j < nc; j += NT) {
      const int ci = ts.cand[j];
      const uint32_t cu = ts.ckey[j];
      int r0 = 0, r1 = 0;
      int m = 0;
      for (; m + 1 < nc; m += 2) {
        const uint32_t a0 = ts.ckey[m], a1 = ts.ckey[m + 1];
        const int c0 = ts.cand[m], c1 = ts.cand[m + 1];
        r0 += (a0 > cu) | ((a0 == cu) & (c0 < ci));
        r1 += (a1 > cu) | ((a1 == cu) & (c1 < ci));
      }
      if (m < nc) r0 += (ts.ckey[m] > cu) | ((ts.ckey[m] == cu) & (ts.cand[m] < ci));
      if (r0 + r1 == need - 1) {
        ts.tkey = cu;
        ts.tidx = ci;
      }
    }
    __syncthreads();
  }
  const uint32_t T = (by_index || all_in) ? lo : ts.tkey;
  const int tI = (by_index || all_in) ? n : ts.tidx;  // all_in: every key >= lo is taken
  // 0: not taken, 1: taken, 2: a boundary key, taken by ascending index
  auto pick = [&](int i) -> int {
    const uint32_t u = key(i);
    if (u > hi) return 1;
    if (u < lo) return 0;
    if (by_index) return 2;
    return (u > T || (u == T && i <= tI)) ? 1 : 0;
  };

  // 4. ascending compaction: counts per thread, one block scan, then the writes
  int c1 = 0, c2 = 0;
#pragma unroll 4
  for (int i = s0; i < s1; ++i) {
    const int t = pick(i);
    c1 += t == 1;
    c2 += t == 2;
  }
  int x1 = c1, x2 = c2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y1 = __shfl_up_sync(0xffffffffu, x1, o), y2 = __shfl_up_sync(0xffffffffu, x2, o);
    if (lane >= o) {
      x1 += y1;
      x2 += y2;
    }
  }
  if (lane == 31) {
    ts.wa[warp] = x1;
    ts.wb[warp] = x2;
  }
  __syncthreads();
  int base = x1 - c1, bseen = x2 - c2;
  for (int w = 0; w < warp; ++w) {
    base += ts.wa[w];
    bseen += ts.wb[w];
  }
  int o = base + min(need, bseen);
  for (int i = s0; i < s1; ++i) {
    const int t = pick(i);
    if (t == 1 || (t == 2 && bseen < need)) {
      if (o < k) take(o, i);
      ++o;
    }
    bseen += t == 2;
  }
  __syncthreads();  // the scratch may be reused right after
}

// topk_adaptive_fn writing the ascending indices to out[0..k) (and out2, when not null).
template <int NT, class KeyFn>
__device__ void topk_adaptive(int n, int k, KeyFn key, TopkSmem<NT>& ts, int32_t* out, int32_t* out2) {
  topk_adaptive_fn<NT>(n, k, key, ts, [&](int pos, int i) {
    out[pos] = i;
    if (out2) out2[pos] = i;
  });
}

// The same selection written without divergent branches in its per-key work: on this
// GPU a data-dependent branch inside an unrolled per-key loop costs on the order of
// a hundred cycles (measured: the compaction's two passes took 4,800 cycles with
// branches and 1,700 with the decisions as bit arithmetic and predicated stores).
// Thread t owns the contiguous keys [t S, t S + S), S a multiple of 4 (16-byte loads,
// index-ordered compaction by one block scan); every thread runs the same trip counts.
// Boundary candidates are gathered by a block scan instead of shared atomics, and the
// gather and the compaction visit only the keys they keep (bit masks of a thread's at
// most 32 keys).  Needs n <= 32 NT, with `keys` 16-byte aligned and readable up to
// NT * S entries (entries from n on are ignored).  For 1 <= k < n; every thread of the
// block calls this.
template <int NT>
__device__ void topk_flat(const uint32_t* keys, int n, int k, TopkSmem<NT>& ts, int32_t* out) {
  static_assert(NT % 32 == 0 && kTkBins % NT == 0 && (kTkBins / NT) % 4 == 0, "bins must split into uint4s");
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int NW = NT / 32;
  constexpr int BPT = kTkBins / NT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = ((n + NT - 1) / NT + 3) & ~3;  // keys per thread
  const int Q = S >> 2;                         // 16-byte groups per thread
  const int i0 = tid * S;
  const uint4* k4 = reinterpret_cast<const uint4*>(keys + i0);
  uint4* h4 = reinterpret_cast<uint4*>(ts.hist);
  for (int j = tid; j < kTkBins / 4; j += NT) h4[j] = make_uint4(0, 0, 0, 0);

  // block-wide exclusive prefix of one int per thread (and the total), by shuffles
  // and one barrier; `slot` picks one of two scratch rows so back-to-back calls do not
  // race
  auto block_scan = [&](int x, int slot, int& total) -> int {
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, o);
      incl += lane >= o ? y : 0;
    }
    int* wsum = slot ? ts.wb : ts.wa;
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = incl - x;
    total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int v = wsum[w];
      before += w < warp ? v : 0;
      total += v;
    }
    return before;
  };

  // 1. the key range
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll 1
  for (int q = 0; q < Q; ++q) {
    const uint4 v = k4[q];
    const int j = i0 + 4 * q;
    lo = min(lo, j < n ? v.x : 0xffffffffu);
    hi = max(hi, j < n ? v.x : 0u);
    lo = min(lo, j + 1 < n ? v.y : 0xffffffffu);
    hi = max(hi, j + 1 < n ? v.y : 0u);
    lo = min(lo, j + 2 < n ? v.z : 0xffffffffu);
    hi = max(hi, j + 2 < n ? v.z : 0u);
    lo = min(lo, j + 3 < n ? v.w : 0xffffffffu);
    hi = max(hi, j + 3 < n ? v.w : 0u);
  }
  lo = __reduce_min_sync(FULL, lo);
  hi = __reduce_max_sync(FULL, hi);
  if (lane == 0) {
    ts.wlo[warp] = lo;
    ts.whi[warp] = hi;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    lo = min(lo, ts.wlo[w]);
    hi = max(hi, ts.whi[w]);
  }

  // 2. shrink [lo, hi]; `need` of the `nin` keys inside it are taken
  int need = k, nin = n;
  bool cleared = true;
  while (nin > kTkCandFlat && lo != hi) {
    if (!cleared) {
      for (int j = tid; j < kTkBins / 4; j += NT) h4[j] = make_uint4(0, 0, 0, 0);
      __syncthreads();
    }
    cleared = false;
    const uint32_t range = hi - lo;
    const int shift = range < (uint32_t)kTkBins ? 0 : (32 - __clz(range)) - 10;
#pragma unroll 1
    for (int q = 0; q < Q; ++q) {
      const uint4 v = k4[q];
      const uint32_t u4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t u = u4[e];
        if ((i0 + 4 * q + e < n) & (u >= lo) & (u <= hi)) atomicAdd(&ts.hist[(u - lo) >> shift], 1u);
      }
    }
    __syncthreads();
    uint32_t c[BPT];
#pragma unroll
    for (int j = 0; j < BPT; j += 4) {
      const uint4 v = h4[(tid * BPT + j) >> 2];
      c[j] = v.x;
      c[j + 1] = v.y;
      c[j + 2] = v.z;
      c[j + 3] = v.w;
    }
    int sum = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) sum += (int)c[j];
    int incl = sum;  // over the lanes >= this one
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(FULL, incl, o);
      incl += lane + o < 32 ? y : 0;
    }
    if (lane == 0) ts.wa[warp] = incl;
    __syncthreads();
    int above = incl - sum;
#pragma unroll
    for (int w = 0; w < NW; ++w) above += w > warp ? ts.wa[w] : 0;
    if (above < need && above + sum >= need) {  // exactly one thread
      int acc = above, bstar = 0, nn = 0, nb = 0;
#pragma unroll
      for (int j = BPT - 1; j >= 0; --j) {
        const bool hit = nb == 0 && acc + (int)c[j] >= need;
        bstar = hit ? tid * BPT + j : bstar;
        nn = hit ? need - acc : nn;
        nb = hit ? (int)c[j] : nb;
        acc += (int)c[j];
      }
      ts.bstar = bstar;
      ts.need = nn;
      ts.nb = nb;
    }
    __syncthreads();
    const uint32_t nlo = lo + ((uint32_t)ts.bstar << shift);
    hi = shift == 0 ? nlo : min(hi, nlo + ((1u << shift) - 1u));
    lo = nlo;
    need = ts.need;
    nin = ts.nb;
    // the next round's first barrier orders these reads before the next writes
  }

  // 3. the boundary pair (T, t) among at most kTkCandFlat candidates, gathered in
  // index order by a block scan and ranked by warps 0 and 1 (one candidate a lane,
  // compared with the others four at a time, over the gathered ones only)
  const bool all_in = need == nin;                    // every key in [lo, hi] is taken
  const bool by_index = !all_in && nin > kTkCandFlat;  // then lo == hi
  if (!by_index && !all_in) {
    // this thread's keys inside [lo, hi] as a bit mask (S <= 32 keys a thread)
    uint32_t fm = 0;
#pragma unroll 1
    for (int q = 0; q < Q; ++q) {
      const uint4 v = k4[q];
      const int j = i0 + 4 * q;
      const uint32_t f = (uint32_t)((j < n) & (v.x >= lo) & (v.x <= hi)) |
                         ((uint32_t)((j + 1 < n) & (v.y >= lo) & (v.y <= hi)) << 1) |
                         ((uint32_t)((j + 2 < n) & (v.z >= lo) & (v.z <= hi)) << 2) |
                         ((uint32_t)((j + 3 < n) & (v.w >= lo) & (v.w <= hi)) << 3);
      fm |= f << (4 * q);
    }
    int total;
    int slot = block_scan(__popc(fm), 0, total);
    while (fm) {  // the few candidates, in index order
      const int e = __ffs(fm) - 1;
      fm &= fm - 1;
      if (slot < kTkCandFlat) {
        ts.cand[slot] = i0 + e;
        ts.ckey[slot] = keys[i0 + e];
      }
      ++slot;
    }
    __syncthreads();
    static_assert(kTkCandFlat <= NT && kTkCandFlat % 32 == 0, "one candidate a lane");
    if (warp < kTkCandFlat / 32) {
      const int nc = nin;  // <= kTkCandFlat here
      const int me = warp * 32 + lane;
      const int ci = me < nc ? ts.cand[me] : 0;
      const uint32_t cu = me < nc ? ts.ckey[me] : 0u;
      const uint4* a4 = reinterpret_cast<const uint4*>(ts.ckey);
      const int4* c4 = reinterpret_cast<const int4*>(ts.cand);
      int r = 0;
#pragma unroll 1
      for (int m4 = 0; m4 < (nc + 3) >> 2; ++m4) {  // entries from nc on are ignored
        const uint4 a = a4[m4];
        const int4 c = c4[m4];
        const int m = 4 * m4;
        r += (m < nc) & ((a.x > cu) | ((a.x == cu) & (c.x < ci)));
        r += (m + 1 < nc) & ((a.y > cu) | ((a.y == cu) & (c.y < ci)));
        r += (m + 2 < nc) & ((a.z > cu) | ((a.z == cu) & (c.z < ci)));
        r += (m + 3 < nc) & ((a.w > cu) | ((a.w == cu) & (c.w < ci)));
      }
      if ((me < nc) & (r == need - 1)) {
        ts.tkey = cu;
        ts.tidx = ci;
      }
    }
    __syncthreads();
  }
  const uint32_t T = (by_index || all_in) ? lo : ts.tkey;
  const int tI = (by_index || all_in) ? n : ts.tidx;  // all_in: every key >= lo is taken
  const unsigned bi = by_index ? 1u : 0u;

  // 4. ascending compaction.  Class bit 0: taken; bit 1: a boundary key taken by index
  // (the first `need` of them in index order).
  auto cls = [&](uint32_t u, int i) -> unsigned {
    const unsigned valid = (unsigned)(i < n);
    const unsigned above = (unsigned)(u > hi);
    const unsigned inr = (unsigned)(u >= lo) & (above ^ 1u);
    const unsigned tk = above | (inr & (bi ^ 1u) & ((unsigned)(u > T) | ((unsigned)(u == T) & (unsigned)(i <= tI))));
    return (0u - valid) & (tk | ((inr & bi) << 1));  // all bits of the class, or none
  };
  // this thread's taken keys (tm) and boundary keys taken by index (bm) as bit masks
  uint32_t tm = 0, bm = 0;
#pragma unroll 1
  for (int q = 0; q < Q; ++q) {
    const uint4 v = k4[q];
    const int j = i0 + 4 * q;
    const unsigned a = cls(v.x, j), b = cls(v.y, j + 1), c = cls(v.z, j + 2), d = cls(v.w, j + 3);
    tm |= ((a & 1u) | ((b & 1u) << 1) | ((c & 1u) << 2) | ((d & 1u) << 3)) << (4 * q);
    bm |= ((a >> 1) | ((b >> 1) << 1) | ((c >> 1) << 2) | ((d >> 1) << 3)) << (4 * q);
  }
  // both prefixes in one scan, one count in each 16-bit half (every count is <= n < 2^16)
  int tot;
  const int both = block_scan(__popc(tm) | (__popc(bm) << 16), 1, tot);
  const int base = both & 0xffff;
  int bseen = both >> 16;
  int o = base + min(need, bseen);
  uint32_t any = tm | bm;
  while (any) {  // this thread's taken keys, in index order
    const int e = __ffs(any) - 1;
    any &= any - 1;
    const unsigned isb = (bm >> e) & 1u;
    const bool take = (isb ^ 1u) | (unsigned)(bseen < need);
    if (take & (o < k)) out[o] = i0 + e;
    o += take;
    bseen += (int)isb;
  }
  __syncthreads();  // the list is complete and the scratch may be reused
}

// Top-k by counting, for up to a few hundred keys.  Key i's rank is the number of keys that
// beat it (larger, or equal at a lower index); i is taken iff its rank is below k, so
// exactly k are taken, ties going to the lower index.  Thread t owns indices t + NT m
// (m < KPT) and compares them with all n keys, read by broadcast 16-byte loads:
// n KPT compares per thread and two barriers, against the several barrier-separated
// passes of the histogram select.  Needs n <= NT KPT and `keys` 16-byte aligned; reads
// keys[0, n) only.  The ascending list goes to out[0..k).  Every thread calls this.
template <int NT, int KPT>
__device__ void topk_rank(const uint32_t* keys, int n, int k, TopkSmem<NT>& ts, int32_t* out) {
  constexpr int NW = NT / 32;
  static_assert(NT % 32 == 0 && KPT * NW <= kTkBins, "counts must fit the histogram scratch");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* cnt = reinterpret_cast<int*>(ts.hist);
  const int n4 = n >> 2;
  uint32_t kv[KPT], km[KPT];
  int rk[KPT], g4[KPT];
#pragma unroll
  for (int m = 0; m < KPT; ++m) {
    const int i = tid + NT * m;
    kv[m] = i < n ? keys[i] : 0u;
    km[m] = kv[m] - 1u;  // j < i beats i iff key_j >= key_i, i.e. key_j > key_i - 1
    rk[m] = 0;
    g4[m] = i >> 2;
  }
  // whole groups of four: groups below i's own compare against key_i - 1
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
#pragma unroll 4
  for (int j4 = 0; j4 < n4; ++j4) {
    const uint4 u = k4[j4];
#pragma unroll
    for (int m = 0; m < KPT; ++m) {
      const uint32_t t = j4 < g4[m] ? km[m] : kv[m];
      rk[m] += ((u.x > t) + (u.y > t)) + ((u.z > t) + (u.w > t));
    }
  }
  bool taken[KPT];
#pragma unroll
  for (int m = 0; m < KPT; ++m) {
    const int i = tid + NT * m;
    taken[m] = false;
    if (i >= n) continue;
    // key_i = 0: key_i - 1 wrapped, so the groups below i's counted nothing; all beat i
    if (kv[m] == 0u) rk[m] += 4 * min(g4[m], n4);
    // i's own group was compared as if it lay above i: add the equal members below i
    if (g4[m] < n4)
      for (int j = 4 * g4[m]; j < i; ++j) rk[m] += keys[j] == kv[m];
    // the last n % 4 keys, one by one
    for (int j = 4 * n4; j < n; ++j) rk[m] += keys[j] > kv[m] || (keys[j] == kv[m] && j < i);
    taken[m] = rk[m] < k;
  }
  // ascending compaction: index order is (m, warp, lane)
  unsigned bal[KPT];
#pragma unroll
  for (int m = 0; m < KPT; ++m) {
    bal[m] = __ballot_sync(0xffffffffu, taken[m]);
    if (lane == 0) cnt[m * NW + warp] = __popc(bal[m]);
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < KPT; ++m) {
    if (taken[m]) {
      int pos = __popc(bal[m] & ((1u << lane) - 1u));
      for (int q = 0; q < m * NW + warp; ++q) pos += cnt[q];
      out[pos] = tid + NT * m;
    }
  }
  __syncthreads();  // the list is complete and the scratch may be reused
}

}  // namespace rkv
