// Stage 2 of RocketKV: one Hybrid Sparse Attention (HSA) decode step.
//
// "RocketKV-adapted -- Two-Stage Compression" (VeloxQuant-MLX docs), section
// "Where it sits -- the mechanism gap": HSA bounds each page's score from
// Quest-style paged element-wise max/min summaries along the sequence, restricted
// to the SparQ-style top-magnitude channels of the query along the head dimension;
// section "Adaptation notes": whole pages (k2 of them) are selected and attended.
//
// Two implementations of the same step:
//
// * hsa_step_kernel (fused, one launch): one thread-block cluster per (sequence, KV
//   head).  Optionally appends the new token first.  Every CTA selects the
//   channels; each CTA stages the summaries of its slice of pages into shared
//   memory with bulk copies (one round trip) and bounds those pages; the page
//   scores are shared through distributed shared memory; every CTA runs the same
//   top-k2 select, attends over its share of the selected pages, and the CTAs'
//   partial softmax states are merged through distributed shared memory.  Used
//   while a layer's page count fits the CTA's shared memory (max_pages <= 4096).
// * hsa_score -> hsa_topk -> hsa_attend -> hsa_combine (four launches, scratch in the
//   caller's workspace) for larger caches.
//
// Attention in both: the selected pages are cut into 16-token chunks; each warp
// streams chunks through a ring of shared-memory stages filled by bulk copies
// (cp.async.bulk, TMA engine; one 256-B row per lane, 16 K rows + 16 V rows) that
// complete on an mbarrier; q.K^T and P.V are m16n8k16 bf16 tensor-core MMAs with
// the GQA group's heads as the M rows; fp32 online softmax; P split into bf16 hi +
// lo so the P.V product keeps ~16 bits of the probabilities.
#include <climits>

#include <cooperative_groups.h>

#include "rkv_device.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

namespace cg = cooperative_groups;

constexpr int kMaxSplit = 64;
constexpr int kScoreThreads = 256;
constexpr int kScorePages = 2 * kScoreThreads;  // pages scored per CTA (2 per thread)
constexpr int kTopkThreads = 1024;
constexpr int kAtWarps = 4;
constexpr int kThreads = kAtWarps * 32;
constexpr int kSplitStages = 3;
constexpr int kFusedStages = 2;
constexpr int kChunkTok = 16;                           // tokens per pipeline stage
constexpr int kRowBytes = 272;                          // 256 B token row + 16 B pad
constexpr int kStageBytes = 2 * kChunkTok * kRowBytes;  // K rows then V rows
constexpr int kWarpCombineBytes = kAtWarps * 8 * (2 + 128) * 4;
constexpr int kFusedMaxPages = 4096;
constexpr int kMaxCluster = 8;

constexpr int ring_bytes(int stages) { return kAtWarps * stages * kStageBytes; }
constexpr int kSplitSmem = ring_bytes(kSplitStages) > kWarpCombineBytes ? ring_bytes(kSplitStages) : kWarpCombineBytes;
static_assert(ring_bytes(kFusedStages) >= kWarpCombineBytes, "the ring doubles as the warp-combine buffer");
// the summary staging tile must hold at least 8 pages of all 128 channels (Kmax + Kmin)
static_assert(ring_bytes(kFusedStages) >= 2 * 128 * 8 * 2, "staging tile too small");

struct HsaParams {
  rkv_bf16* k_pages;
  rkv_bf16* v_pages;
  const int32_t* page_table;
  int32_t* seq_len;
  rkv_bf16* kmax;
  rkv_bf16* kmin;
  int32_t* err;
  int32_t* sync;           // [B] arrival counters (fused step with append)
  const rkv_bf16* q;
  const rkv_bf16* k_new;   // [B][Hkv][128] or null (no append)
  const rkv_bf16* v_new;
  float* sigma;            // [units][max_pages]      (split path)
  int32_t* selp;           // [units][max_pages]      (split path)
  float* part_o;           // [B*Hq][nsplit][128]     (split path)
  float2* part_ml;         // [B*Hq][nsplit]          (split path)
  float* out;              // [B*Hq][128]
  int32_t* sel_channels;
  int32_t* sel_pages;
  int sel_pages_stride;
  int B, Hkv, Hq, G, P, max_pages, num_phys, nsplit, cluster;
  float scale_log2;
  int32_t k1[RKV_MAX_BATCH];
  int32_t k2[RKV_MAX_BATCH];
};

// Current length of sequence b, clamped to the cache capacity (flagging overflow).
__device__ __forceinline__ int seq_length(const HsaParams& p, int b) {
  int n = p.seq_len[b];
  const int cap = p.max_pages * p.P;
  if (n < 0 || n > cap) {
    flag_error(p.err, RKV_DEVERR_CAPACITY);
    n = n < 0 ? 0 : cap;
  }
  return n;
}

// Shared-memory state of the channel selection (one KV head).
struct ChanSmem {
  float qf[8][128];
  unsigned long long akey[128];
  int chan[128];
  float qpos[128], qneg[128];
  int warp_cnt[4];
};

// Top-k1 channels of a_i = sum_h |q_h,i| (ties: lower channel), ascending, with the
// per-channel sums of the positive and negative parts of q over the group.  The
// channel score is summed in fp64, where a sum of <= 8 bf16 magnitudes is exact, and
// ranked on its bit pattern (order-preserving for non-negative doubles).
// Every thread of a block of >= 128 threads calls this after filling qf.
__device__ void select_channels(ChanSmem& cs, int G, int k1) {
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid < 128) {
    double s = 0.0;
    for (int h = 0; h < G; ++h) s += fabs((double)cs.qf[h][tid]);
    cs.akey[tid] = (unsigned long long)__double_as_longlong(s);
  }
  __syncthreads();
  bool sel = false;
  unsigned bal = 0;
  if (tid < 128) {
    const unsigned long long ai = cs.akey[tid];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < 128; ++j) {
      const unsigned long long aj = cs.akey[j];
      rank += (aj > ai) || (aj == ai && j < tid);
    }
    sel = rank < k1;
    bal = __ballot_sync(0xffffffffu, sel);
    if ((tid & 31) == 0) cs.warp_cnt[tid >> 5] = __popc(bal);
  }
  __syncthreads();
  if (tid < 128 && sel) {
    int pos = __popc(bal & ((1u << (tid & 31)) - 1u));
    for (int w = 0; w < (tid >> 5); ++w) pos += cs.warp_cnt[w];
    cs.chan[pos] = tid;
    float sp = 0.f, sn = 0.f;
    for (int h = 0; h < G; ++h) {
      const float x = cs.qf[h][tid];
      sp += fmaxf(x, 0.f);
      sn += fminf(x, 0.f);
    }
    cs.qpos[pos] = sp;
    cs.qneg[pos] = sn;
  }
  __syncthreads();
}

// Bound of pages pg and pg+1 (pg even) of unit `unit` over the selected channels,
// read straight from global memory:
// s_p = sum_i Kmax_i,p * qpos_i + Kmin_i,p * qneg_i, which equals
// sum_h sum_i max(q_h,i Kmax_i,p, q_h,i Kmin_i,p) since the max picks Kmax for q >= 0.
__device__ __forceinline__ float2 page_pair_bound(const HsaParams& p, int unit, int pg, int k1, const ChanSmem& cs) {
  const size_t base = (size_t)unit * 128 * p.max_pages + pg;
  const unsigned int* mxp = reinterpret_cast<const unsigned int*>(p.kmax + base);
  const unsigned int* mnp = reinterpret_cast<const unsigned int*>(p.kmin + base);
  const int hs = p.max_pages >> 1;  // row stride in bf16 pairs
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
  for (int kk = 0; kk < k1; ++kk) {
    const size_t off = (size_t)cs.chan[kk] * hs;
    const uint32_t hi = __ldg(mxp + off);
    const uint32_t lo = __ldg(mnp + off);
    const float qp = cs.qpos[kk], qn = cs.qneg[kk];
    s0 = fmaf(qp, bf16_lo(hi), s0);
    s0 = fmaf(qn, bf16_lo(lo), s0);
    s1 = fmaf(qp, bf16_hi(hi), s1);
    s1 = fmaf(qn, bf16_hi(lo), s1);
  }
  return make_float2(s0, s1);
}

// Writes the ascending indices of the top-k of keys[0..n) (1 <= k < n) to out[0..k):
// every key > T, and keys == T by ascending index until k are taken.
template <int NT>
__device__ void topk_ascending(const uint32_t* keys, int n, int k, uint32_t* hist, int* scan, int32_t* out,
                               int32_t* out2) {
  uint32_t T;
  int need;
  block_radix_threshold<NT>(n, k, [&](int i) { return keys[i]; }, hist, &T, &need);
  const int tid = threadIdx.x;
  const int seg = (n + NT - 1) / NT;
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  int ceq = 0;
  for (int i = s0; i < s1; ++i) ceq += keys[i] == T;
  int total;
  const int eq_base = block_exclusive_scan<NT>(ceq, scan, &total);
  int csel = 0;
  for (int i = s0, er = eq_base; i < s1; ++i) {
    const uint32_t u = keys[i];
    if (u > T) ++csel;
    else if (u == T) { csel += er < need; ++er; }
  }
  const int out_base = block_exclusive_scan<NT>(csel, scan, &total);
  for (int i = s0, er = eq_base, o = out_base; i < s1; ++i) {
    const uint32_t u = keys[i];
    bool take = u > T;
    if (u == T) { take = er < need; ++er; }
    if (take && o < k) {
      out[o] = i;
      if (out2) out2[o] = i;
      ++o;
    }
  }
}

// Shared-memory state of one CTA's attention.
template <int STAGES>
struct AttnSmem {
  uint64_t bars[kAtWarps][STAGES];
  int tstart[kAtWarps][STAGES];
  float ctaM[8], ctaL[8];
  float ctaO[8][128];
};

// Attention of one CTA (4 warps) over items [it0, it1) of the unit's selected pages
// `sel` (ascending page ids; item i = chunk i % cpp of page sel[i / cpp]); `ptab` is
// the sequence's page-table row.  Leaves the CTA's merged softmax state per head in
// a.ctaM / a.ctaL / a.ctaO (unnormalised) and returns 1 when a bounded wait ran out.
// `ring` is ring_bytes(STAGES) of shared memory, at least kWarpCombineBytes.
template <int STAGES>
__device__ int attend_cta(const HsaParams& p, const int32_t* sel, const int32_t* ptab, int b, int g, int n, int it0,
                          int it1, uint8_t* ring, AttnSmem<STAGES>& a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.P, G = p.G;
  const int NP = (n + P - 1) / P;
  const int cpp = P / kChunkTok;
  const int mine = it1 - it0 - warp;
  const int nj = mine > 0 ? (mine + kAtWarps - 1) / kAtWarps : 0;
  uint8_t* wbuf = ring + warp * (STAGES * kStageBytes);

  const int hrow = lane >> 2, q4 = lane & 3;
  const bool hv = hrow < G;
  const rkv_bf16* qrow = p.q + ((size_t)b * p.Hq + (size_t)g * G + (hv ? hrow : 0)) * 128;
  uint32_t qa0[8], qa2[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    qa0[kk] = hv ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * q4) : 0u;
    qa2[kk] = hv ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * q4) : 0u;
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&a.bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int j) {
    const int s = j % STAGES;
    const int it = it0 + warp + j * kAtWarps;
    int page = sel[it / cpp];
    const int chunk = it % cpp;
    const bool page_ok = page >= 0 && page < NP;  // always true for the select's output
    page = page_ok ? page : 0;
    int phys = ptab[page];
    int t0 = page * P + chunk * kChunkTok;
    if (!page_ok || phys < 0 || phys >= p.num_phys) {
      flag_error(p.err, RKV_DEVERR_PAGE_ID);
      phys = 0;
      t0 = INT_MAX / 2;  // every token of this chunk is masked
    }
    const size_t off = (((size_t)phys * p.Hkv + g) * P + (size_t)chunk * kChunkTok) * 128;
    if (lane == 0) {
      a.tstart[warp][s] = t0;
      mbar_arrive_expect_tx(&a.bars[warp][s], 2 * kChunkTok * 256);
    }
    __syncwarp();
    const rkv_bf16* src = lane < 16 ? p.k_pages + off + lane * 128 : p.v_pages + off + (lane - 16) * 128;
    bulk_g2s(wbuf + s * kStageBytes + lane * kRowBytes, src, 256, &a.bars[warp][s]);
  };

  float m_run = -1e30f, l_run = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int pre = min(nj, STAGES);
  for (int j = 0; j < pre; ++j) issue(j);
  int issued = pre, consumed = 0, timed_out = 0;
  const float sl = p.scale_log2;
  for (int j = 0; j < nj; ++j) {
    const int s = j % STAGES;
    if (!mbar_wait(&a.bars[warp][s], (uint32_t)((j / STAGES) & 1))) {
      flag_error(p.err, RKV_DEVERR_TIMEOUT);
      timed_out = 1;
      break;
    }
    uint8_t* kb = wbuf + s * kStageBytes;
    uint8_t* vb = kb + kChunkTok * kRowBytes;
    const int nvalid = n - a.tstart[warp][s];
    if (nvalid < kChunkTok) {
      // rows past the end of the sequence hold stale data: zero their V rows
      const int nv = max(nvalid, 0);
      for (int w16 = lane; w16 < (kChunkTok - nv) * 16; w16 += 32)
        *reinterpret_cast<uint4*>(vb + (nv + (w16 >> 4)) * kRowBytes + (w16 & 15) * 16) = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      __syncwarp();
    }
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    const uint32_t kb32 = smem_u32(kb), vb32 = smem_u32(vb);
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, kb32 + (nt * 8 + (lane & 7)) * kRowBytes + (kk2 * 32 + (lane >> 3) * 8) * 2);
        mma_16816(sacc[nt], qa0[2 * kk2], 0u, qa2[2 * kk2], 0u, b0, b1);
        mma_16816(sacc[nt], qa0[2 * kk2 + 1], 0u, qa2[2 * kk2 + 1], 0u, b2, b3);
      }
    }
    const int c0 = 2 * q4;
    const float z0 = (c0 < nvalid) ? sacc[0][0] * sl : -INFINITY;
    const float z1 = (c0 + 1 < nvalid) ? sacc[0][1] * sl : -INFINITY;
    const float z2 = (c0 + 8 < nvalid) ? sacc[1][0] * sl : -INFINITY;
    const float z3 = (c0 + 9 < nvalid) ? sacc[1][1] * sl : -INFINITY;
    float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float alpha = exp2f(m_run - m_new);
    const float p0 = exp2f(z0 - m_new), p1 = exp2f(z1 - m_new);
    const float p2 = exp2f(z2 - m_new), p3 = exp2f(z3 - m_new);
    l_run = l_run * alpha + ((p0 + p1) + (p2 + p3));
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= alpha;
      o[i][1] *= alpha;
    }
    const uint32_t ph0 = pack_bf16x2(p0, p1), ph2 = pack_bf16x2(p2, p3);
    const uint32_t pl0 = pack_bf16x2(p0 - bf16_lo(ph0), p1 - bf16_hi(ph0));
    const uint32_t pl2 = pack_bf16x2(p2 - bf16_lo(ph2), p3 - bf16_hi(ph2));
#pragma unroll
    for (int nt2 = 0; nt2 < 8; ++nt2) {
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(v0, v1, v2, v3,
                vb32 + ((lane & 7) + ((lane >> 3) & 1) * 8) * kRowBytes + (nt2 * 16 + (lane >> 4) * 8) * 2);
      mma_16816(o[2 * nt2], ph0, 0u, ph2, 0u, v0, v1);
      mma_16816(o[2 * nt2], pl0, 0u, pl2, 0u, v0, v1);
      mma_16816(o[2 * nt2 + 1], ph0, 0u, ph2, 0u, v2, v3);
      mma_16816(o[2 * nt2 + 1], pl0, 0u, pl2, 0u, v2, v3);
    }
    __syncwarp();
    consumed = j + 1;
    if (j + STAGES < nj) {
      issue(j + STAGES);
      issued = j + STAGES + 1;
    }
  }
  if (timed_out) {
    // wait (bounded) for this warp's copies still in flight before the ring is reused
    for (int j = consumed; j < issued; ++j) mbar_wait(&a.bars[warp][j % STAGES], (uint32_t)((j / STAGES) & 1));
  }
  const int any_to = __syncthreads_or(timed_out);

  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  float* cm = reinterpret_cast<float*>(ring);  // the ring is free now
  float* cl = cm + kAtWarps * 8;
  float* co = cl + kAtWarps * 8;
  if (hv) {
    if (q4 == 0) {
      cm[warp * 8 + hrow] = m_run;
      cl[warp * 8 + hrow] = l_run;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      co[(warp * 8 + hrow) * 128 + nt * 8 + 2 * q4] = o[nt][0];
      co[(warp * 8 + hrow) * 128 + nt * 8 + 2 * q4 + 1] = o[nt][1];
    }
  }
  __syncthreads();
  const int c = threadIdx.x;
  for (int h = 0; h < G; ++h) {
    float M = -1e30f;
#pragma unroll
    for (int w = 0; w < kAtWarps; ++w) M = fmaxf(M, cm[w * 8 + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kAtWarps; ++w) {
      const float f = exp2f(cm[w * 8 + h] - M);
      L += cl[w * 8 + h] * f;
      O += co[(w * 8 + h) * 128 + c] * f;
    }
    a.ctaO[h][c] = O;
    if (c == 0) {
      a.ctaM[h] = M;
      a.ctaL[h] = L;
    }
  }
  __syncthreads();
  return any_to;
}

// ---------------------------------------------------------------------------
// Fused decode step.  grid (C, B*Hkv), cluster (C, 1, 1), 128 threads.
// Dynamic shared memory: ring (2 stages x 4 warps; first used to stage summaries) |
// keys [max_pages] | sel [max_pages] | page-table row [max_pages].
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) hsa_step_kernel(const __grid_constant__ HsaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ ChanSmem cs;
  __shared__ AttnSmem<kFusedStages> as;
  __shared__ uint32_t hist[258];
  __shared__ int scan[kAtWarps + 1];
  __shared__ uint64_t sbar, pbar;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = p.cluster;
  const int rank = (int)cluster.block_rank();
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x;
  const int G = p.G, P = p.P;
  uint8_t* ring = smem;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + ring_bytes(kFusedStages));
  int32_t* sel = reinterpret_cast<int32_t*>(keys + p.max_pages);
  int32_t* ptab = sel + p.max_pages;

  // 1. length before this step; the append makes it n0 + 1
  const int cap = p.max_pages * P;
  int n0 = p.seq_len[b];
  bool do_append = p.k_new != nullptr;
  if (n0 < 0 || n0 + (do_append ? 1 : 0) > cap) {
    if (rank == 0 && tid == 0) flag_error(p.err, RKV_DEVERR_CAPACITY);
    n0 = n0 < 0 ? 0 : (n0 > cap ? cap : n0);
    do_append = false;
  }
  const int n = n0 + (do_append ? 1 : 0);
  const int NP = (n + P - 1) / P;

  // 2. barriers; prefetch of the sequence's page-table row (needed after the select)
  if (tid == 0) {
    mbar_init(&sbar, 1);
    mbar_init(&pbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int np4 = ((NP + 3) & ~3);  // whole 16-byte groups; within the row (max_pages % 8 == 0)
  if (tid == 0) {
    if (np4 > 0) {
      mbar_arrive_expect_tx(&pbar, (uint32_t)np4 * 4);
      bulk_g2s(ptab, p.page_table + (size_t)b * p.max_pages, (uint32_t)np4 * 4, &pbar);
    } else {
      mbar_arrive_expect_tx(&pbar, 0);
    }
  }

  // 3. query of the group
  const rkv_bf16* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128;
  for (int i = tid; i < G * 128; i += kThreads) cs.qf[i >> 7][i & 127] = bf16_f(qg[i]);

  // 4. append (rank 0): token into its slot, its page's Kmax/Kmin folded
  if (do_append && rank == 0 && tid < 64) {
    const int page = n0 / P, slot = n0 % P;
    const int phys = p.page_table[(size_t)b * p.max_pages + page];
    if (phys >= 0 && phys < p.num_phys) {
      const size_t src = ((size_t)b * p.Hkv + g) * 128 + 2 * tid;
      const size_t dst = (((size_t)phys * p.Hkv + g) * P + slot) * 128 + 2 * tid;
      const uint32_t ku = *reinterpret_cast<const uint32_t*>(p.k_new + src);
      *reinterpret_cast<uint32_t*>(p.k_pages + dst) = ku;
      *reinterpret_cast<uint32_t*>(p.v_pages + dst) = *reinterpret_cast<const uint32_t*>(p.v_new + src);
      const size_t row = ((size_t)unit * 128 + 2 * tid) * p.max_pages + page;
      float mx0 = bf16_lo(ku), mx1 = bf16_hi(ku), mn0 = mx0, mn1 = mx1;
      if (slot > 0) {
        mx0 = fmaxf(bf16_f(p.kmax[row]), mx0);
        mx1 = fmaxf(bf16_f(p.kmax[row + p.max_pages]), mx1);
        mn0 = fminf(bf16_f(p.kmin[row]), mn0);
        mn1 = fminf(bf16_f(p.kmin[row + p.max_pages]), mn1);
      }
      p.kmax[row] = (rkv_bf16)(__float_as_uint(mx0) >> 16);
      p.kmax[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mx1) >> 16);
      p.kmin[row] = (rkv_bf16)(__float_as_uint(mn0) >> 16);
      p.kmin[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mn1) >> 16);
      // the new K/V row and summaries are read back by bulk copies (async proxy)
      asm volatile("fence.proxy.async.global;\n" ::: "memory");
    } else {
      flag_error(p.err, RKV_DEVERR_PAGE_ID);
    }
  }

  // 5. channels (every CTA)
  const int k1 = p.k1[b];
  select_channels(cs, G, k1);
  cluster.sync();  // the append is visible; every CTA of the cluster has read seq_len

  // 6. the last cluster of sequence b to get here advances seq_len
  if (do_append && rank == 0 && tid == 0) {
    __threadfence();
    if (atomicAdd(&p.sync[b], 1) == p.Hkv - 1) {
      p.sync[b] = 0;
      p.seq_len[b] = n;
    }
  }

  // 7. page bounds of this CTA's slice [p0, p1) (8-page aligned).  The k1 Kmax and
  // k1 Kmin row pieces of a tile are bulk-copied into the ring at once (one round
  // trip), then every thread bounds pages from shared memory.
  const int per = ((NP + C - 1) / C + 7) & ~7;
  const int p0 = min(NP, rank * per), p1 = min(NP, p0 + per);
  const int tcap = (ring_bytes(kFusedStages) / (4 * k1)) & ~7;
  const rkv_bf16* smax = reinterpret_cast<const rkv_bf16*>(ring);
  for (int t0 = p0, tile = 0; t0 < p1; t0 += tcap, ++tile) {
    const int cnt = min(tcap, p1 - t0);
    const int cnt8 = (cnt + 7) & ~7;  // t0 + cnt8 <= max_pages since both are multiples of 8
    fence_proxy_async_smem();
    __syncthreads();  // the previous tile is consumed
    if (tid == 0) mbar_arrive_expect_tx(&sbar, (uint32_t)(2 * k1 * cnt8 * 2));
    __syncthreads();
    for (int i = tid; i < 2 * k1; i += kThreads) {
      const rkv_bf16* base = i < k1 ? p.kmax : p.kmin;
      const int ch = cs.chan[i < k1 ? i : i - k1];
      bulk_g2s(ring + (size_t)i * cnt8 * 2, base + ((size_t)unit * 128 + ch) * p.max_pages + t0,
               (uint32_t)cnt8 * 2, &sbar);
    }
    if (!mbar_wait(&sbar, (uint32_t)(tile & 1))) flag_error(p.err, RKV_DEVERR_TIMEOUT);
    for (int j = tid; j < cnt; j += kThreads) {
      float s = 0.f;
      for (int kk = 0; kk < k1; ++kk) {
        s = fmaf(cs.qpos[kk], bf16_f(smax[kk * cnt8 + j]), s);
        s = fmaf(cs.qneg[kk], bf16_f(smax[(k1 + kk) * cnt8 + j]), s);
      }
      keys[t0 + j] = float_key(s);
    }
  }
  fence_proxy_async_smem();  // generic reads of the ring before the attention's bulk copies
  cluster.sync();            // every slice is written

  // 8. gather the other slices, then the same top-k2 in every CTA
  for (int r = 0; r < C; ++r) {
    if (r == rank) continue;
    const uint32_t* remote = cluster.map_shared_rank(keys, r);
    const int r0 = min(NP, r * per), r1 = min(NP, r0 + per);
    for (int i = r0 + tid; i < r1; i += kThreads) keys[i] = remote[i];
  }
  __syncthreads();
  const int k = min(p.k2[b], NP);
  int32_t* user_pages = (rank == 0 && p.sel_pages) ? p.sel_pages + (size_t)unit * p.sel_pages_stride : nullptr;
  if (k >= NP) {
    for (int i = tid; i < NP; i += kThreads) {
      sel[i] = i;
      if (user_pages) user_pages[i] = i;
    }
  } else {
    topk_ascending<kThreads>(keys, NP, k, hist, scan, sel, user_pages);
  }
  if (user_pages && tid == 0 && k < p.sel_pages_stride) user_pages[k] = -1;
  if (rank == 0 && p.sel_channels && tid < 128) p.sel_channels[(size_t)unit * 128 + tid] = tid < k1 ? cs.chan[tid] : -1;
  if (!mbar_wait(&pbar, 0)) flag_error(p.err, RKV_DEVERR_TIMEOUT);
  __syncthreads();

  // 9. attention over this CTA's share of the selected chunks
  const int items = k * (P / kChunkTok);
  const int ips = (items + C - 1) / C;
  const int it0 = min(items, rank * ips), it1 = min(items, it0 + ips);
  attend_cta<kFusedStages>(p, sel, ptab, b, g, n, it0, it1, ring, as);
  cluster.sync();  // every CTA's partial state is in its shared memory

  // 10. merge the CTAs' states; CTA r finishes heads r, r + C, ...
  for (int h = rank; h < G; h += C) {
    float M = -1e30f;
    for (int r = 0; r < C; ++r) M = fmaxf(M, cluster.map_shared_rank(&as, r)->ctaM[h]);
    float L = 0.f, O = 0.f;
    for (int r = 0; r < C; ++r) {
      const AttnSmem<kFusedStages>* ra = cluster.map_shared_rank(&as, r);
      const float f = exp2f(ra->ctaM[h] - M);
      L += ra->ctaL[h] * f;
      O += ra->ctaO[h][tid] * f;
    }
    p.out[((size_t)b * p.Hq + (size_t)g * G + h) * 128 + tid] = L > 0.f ? O / L : 0.f;
  }
  cluster.sync();  // no CTA leaves while others still read its shared memory
}

// ---------------------------------------------------------------------------
// Split path, steps 1-2: channel selection and page bounds into the workspace.
// grid (ceil(max_pages / 512), B*Hkv), 256 threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScoreThreads) hsa_score_kernel(const __grid_constant__ HsaParams p) {
  __shared__ ChanSmem cs;
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x;
  const int n = seq_length(p, b);
  const int NP = (n + p.P - 1) / p.P;
  const int page0 = blockIdx.x * kScorePages;
  const bool write_ch = (blockIdx.x == 0) && (p.sel_channels != nullptr);
  if (page0 >= NP && !write_ch) return;
  const int G = p.G;
  const rkv_bf16* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128;
  for (int i = tid; i < G * 128; i += kScoreThreads) cs.qf[i >> 7][i & 127] = bf16_f(qg[i]);
  const int k1 = p.k1[b];
  select_channels(cs, G, k1);
  if (write_ch && tid < 128) p.sel_channels[(size_t)unit * 128 + tid] = tid < k1 ? cs.chan[tid] : -1;
  const int pg = page0 + 2 * tid;
  if (pg < NP) {
    const float2 s = page_pair_bound(p, unit, pg, k1, cs);
    float* sg = p.sigma + (size_t)unit * p.max_pages;
    sg[pg] = s.x;
    if (pg + 1 < NP) sg[pg + 1] = s.y;
  }
}

// Split path, step 3: top-k2 pages, ascending.  grid B*Hkv, 1024 threads,
// dynamic shared memory = max_pages keys.
__global__ void __launch_bounds__(kTopkThreads) hsa_topk_kernel(const __grid_constant__ HsaParams p) {
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[258];
  __shared__ int scan_scratch[kTopkThreads / 32 + 1];
  const int unit = blockIdx.x, b = unit / p.Hkv;
  const int tid = threadIdx.x;
  const int n = seq_length(p, b);
  const int NP = (n + p.P - 1) / p.P;
  const int k = min(p.k2[b], NP);
  int32_t* out = p.selp + (size_t)unit * p.max_pages;
  int32_t* user = p.sel_pages ? p.sel_pages + (size_t)unit * p.sel_pages_stride : nullptr;
  if (user && tid == 0 && k < p.sel_pages_stride) user[k] = -1;
  if (k >= NP) {
    for (int i = tid; i < NP; i += kTopkThreads) {
      out[i] = i;
      if (user) user[i] = i;
    }
    return;
  }
  const float* sg = p.sigma + (size_t)unit * p.max_pages;
  for (int i = tid; i < NP; i += kTopkThreads) keys[i] = float_key(sg[i]);
  __syncthreads();
  topk_ascending<kTopkThreads>(keys, NP, k, hist, scan_scratch, out, user);
}

// Split path, step 4: attention over a range of the selected chunks.
// grid (nsplit, B*Hkv), 128 threads.
__global__ void __launch_bounds__(kThreads) hsa_attend_kernel(const __grid_constant__ HsaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ AttnSmem<kSplitStages> as;
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv, split = blockIdx.x;
  const int n = seq_length(p, b);
  const int NP = (n + p.P - 1) / p.P;
  const int k = min(p.k2[b], NP);
  const int items = k * (p.P / kChunkTok);
  const int ips = (items + p.nsplit - 1) / p.nsplit;
  const int it0 = min(items, split * ips), it1 = min(items, it0 + ips);
  if (attend_cta<kSplitStages>(p, p.selp + (size_t)unit * p.max_pages, p.page_table + (size_t)b * p.max_pages, b, g,
                               n, it0, it1, smem, as))
    return;
  const int c = threadIdx.x;
  for (int h = 0; h < p.G; ++h) {
    const size_t bh = (size_t)b * p.Hq + (size_t)g * p.G + h;
    if (p.nsplit == 1) {
      p.out[bh * 128 + c] = as.ctaL[h] > 0.f ? as.ctaO[h][c] / as.ctaL[h] : 0.f;
    } else {
      p.part_o[(bh * p.nsplit + split) * 128 + c] = as.ctaO[h][c];
      if (c == 0) p.part_ml[bh * p.nsplit + split] = make_float2(as.ctaM[h], as.ctaL[h]);
    }
  }
}

// Split path: merge of the splits.  grid B*Hq, 128 threads (one per channel).
__global__ void __launch_bounds__(128) hsa_combine_kernel(const __grid_constant__ HsaParams p) {
  const size_t bh = blockIdx.x;
  const int c = threadIdx.x;
  const float2* ml = p.part_ml + bh * p.nsplit;
  float M = -1e30f;
  for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, ml[s].x);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < p.nsplit; ++s) {
    const float f = exp2f(ml[s].x - M);
    L += ml[s].y * f;
    O += p.part_o[(bh * p.nsplit + s) * 128 + c] * f;
  }
  p.out[bh * 128 + c] = L > 0.f ? O / L : 0.f;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

HsaParams make_params(const DecodeArgs& a) {
  const rkv_cache& c = a.cache;
  HsaParams p;
  p.k_pages = c.k_pages;
  p.v_pages = c.v_pages;
  p.page_table = c.page_table;
  p.seq_len = c.seq_len;
  p.kmax = c.kmax;
  p.kmin = c.kmin;
  p.err = c.error_word;
  p.sync = c.step_sync;
  p.q = a.q;
  p.k_new = a.k_new;
  p.v_new = a.v_new;
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  const size_t units = (size_t)c.B * c.Hkv;
  const size_t sg = align256(units * c.max_pages * 4);
  p.sigma = w ? reinterpret_cast<float*>(w) : nullptr;
  p.selp = w ? reinterpret_cast<int32_t*>(w + sg) : nullptr;
  p.part_o = w ? reinterpret_cast<float*>(w + 2 * sg) : nullptr;
  p.part_ml = w ? reinterpret_cast<float2*>(w + 2 * sg + align256((size_t)c.B * a.Hq * kMaxSplit * 128 * 4)) : nullptr;
  p.out = a.out;
  p.sel_channels = a.sel_channels;
  p.sel_pages = a.sel_pages;
  p.sel_pages_stride = a.sel_pages_stride;
  p.B = c.B;
  p.Hkv = c.Hkv;
  p.Hq = a.Hq;
  p.G = a.G;
  p.P = c.page_size;
  p.max_pages = c.max_pages;
  p.num_phys = c.num_phys_pages;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  for (int b = 0; b < c.B; ++b) {
    p.k1[b] = a.k1[b];
    p.k2[b] = a.k2[b];
  }
  p.nsplit = 1;
  p.cluster = 1;
  return p;
}

int max_items(const DecodeArgs& a) {
  int k2max = 1;
  for (int b = 0; b < a.cache.B; ++b) k2max = a.k2[b] > k2max ? a.k2[b] : k2max;
  return (k2max < a.cache.max_pages ? k2max : a.cache.max_pages) * (a.cache.page_size / kChunkTok);
}

size_t fused_smem_bytes(int max_pages) { return (size_t)ring_bytes(kFusedStages) + 3 * (size_t)max_pages * 4; }

cudaError_t launch_fused(HsaParams& p, const DecodeArgs& a, cudaStream_t s) {
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(hsa_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)fused_smem_bytes(kFusedMaxPages));
    attrs = true;
  }
  const size_t smem = fused_smem_bytes(a.cache.max_pages);
  // CTAs per unit: enough to give every unit a share of one wave of resident CTAs,
  // at most one CTA per 4 attention chunks and at most 8 (a portable cluster)
  static size_t occ_smem = 0;
  static int occ_blocks = 0;
  if (occ_smem != smem) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, hsa_step_kernel, kThreads, smem) != cudaSuccess || nb < 1)
      nb = 1;
    occ_blocks = nb;
    occ_smem = smem;
  }
  const int units = a.cache.B * a.cache.Hkv;
  const int slots = occ_blocks * num_sms();
  int C = units < slots ? slots / units : 1;
  const int by_items = (max_items(a) + kAtWarps - 1) / kAtWarps;
  C = C < by_items ? C : by_items;
  C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
  p.cluster = C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, (unsigned)units, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  launch_begin(K_HSA_STEP, s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, hsa_step_kernel, p);
  launch_end(K_HSA_STEP, s);
  return e;
}

cudaError_t launch_split(HsaParams& p, const DecodeArgs& a, cudaStream_t s) {
  const rkv_cache& c = a.cache;
  const size_t units = (size_t)c.B * c.Hkv;
  const int items = max_items(a);
  int nsplit = (4 * num_sms() + (int)units - 1) / (int)units;
  const int by_items = (items + kAtWarps - 1) / kAtWarps;
  nsplit = nsplit < by_items ? nsplit : by_items;
  nsplit = nsplit < 1 ? 1 : (nsplit > kMaxSplit ? kMaxSplit : nsplit);
  p.nsplit = nsplit;
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(hsa_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmem);
    cudaFuncSetAttribute(hsa_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4);
    attrs = true;
  }
  launch_begin(K_HSA_SCORE, s);
  hsa_score_kernel<<<dim3((c.max_pages + kScorePages - 1) / kScorePages, (unsigned)units), kScoreThreads, 0, s>>>(p);
  launch_end(K_HSA_SCORE, s);
  launch_begin(K_HSA_TOPK, s);
  hsa_topk_kernel<<<(unsigned)units, kTopkThreads, (size_t)c.max_pages * 4, s>>>(p);
  launch_end(K_HSA_TOPK, s);
  launch_begin(K_HSA_ATTEND, s);
  hsa_attend_kernel<<<dim3(nsplit, (unsigned)units), kThreads, kSplitSmem, s>>>(p);
  launch_end(K_HSA_ATTEND, s);
  if (nsplit > 1) {
    launch_begin(K_HSA_COMBINE, s);
    hsa_combine_kernel<<<(unsigned)(c.B * a.Hq), 128, 0, s>>>(p);
    launch_end(K_HSA_COMBINE, s);
  }
  return cudaGetLastError();
}

}  // namespace

size_t decode_ws_bytes(int B, int Hq, int Hkv, int max_pages) {
  const size_t units = (size_t)B * Hkv;
  return align256(units * max_pages * 4) * 2 + align256((size_t)B * Hq * kMaxSplit * 128 * 4) +
         align256((size_t)B * Hq * kMaxSplit * 8);
}

bool decode_fused_ok(const rkv_cache& c) { return c.max_pages <= kFusedMaxPages; }

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  HsaParams p = make_params(a);
  if (a.mode != DECODE_SPLIT && decode_fused_ok(a.cache)) {
    const cudaError_t e = launch_fused(p, a, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  if (a.k_new) {
    const cudaError_t e = launch_append(a.cache, a.k_new, a.v_new, 1, s);
    if (e != cudaSuccess) return e;
    p.k_new = p.v_new = nullptr;
  }
  return launch_split(p, a, s);
}

}  // namespace rkv
