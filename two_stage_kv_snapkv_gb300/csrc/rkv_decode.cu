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
//   head).  Optionally appends the new token (every CTA takes it from shared memory
//   within the step; its K/V and summary updates are stored at the end).  Every CTA
//   selects the channels; each CTA stages the summaries of its slice of pages into
//   shared memory (all channels early for short slices, the chosen ones after the
//   select for long slices: two compiled instances) and bounds those pages; the page
//   scores are shared through distributed shared memory; every CTA runs the same
//   top-k2 select, attends over its share of the selected pages, and the CTAs'
//   partial softmax states are merged through distributed shared memory.  Used
//   while a layer's page count fits the CTA's shared memory (max_pages <= 4096).
// * hsa_score -> hsa_topk -> hsa_attend -> hsa_combine (four launches, scratch in the
//   caller's workspace) for larger caches.
//
// Attention in both: the selected pages are cut into 16-token chunks; each warp
// streams chunks through a ring of shared-memory stages filled by tiled TMA loads
// (cp.async.bulk.tensor, 128-byte swizzle: four 16 x 64 boxes per chunk, K and V
// halves) that complete on an mbarrier; q.K^T and P.V are m16n8k16 bf16 tensor-core
// MMAs fed by ldmatrix from the swizzled rows, with the GQA group's heads as the M
// rows; fp32 online softmax; P split into bf16 hi + lo so the P.V product keeps
// ~16 bits of the probabilities.
#include <climits>
#include <cstddef>
#include <cstring>
#include <type_traits>

#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

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
// instances of the fused step (see hsa_step_kernel)
constexpr int kStepShortRank = 0, kStepShortFlat = 1, kStepLong = 2;
constexpr int kChunkTok = 16;                 // tokens per pipeline stage
constexpr int kHalfBytes = kChunkTok * 128;   // one 16-token x 64-channel box (128-B rows)
constexpr int kStageBytes = 4 * kHalfBytes;   // K lo, K hi, V lo, V hi
constexpr int kWarpCombineBytes = kAtWarps * 8 * (2 + 128) * 4;
constexpr int kFusedMaxPages = 4096;
constexpr int kMaxCluster = 8;

constexpr int ring_bytes(int stages) { return kAtWarps * stages * kStageBytes; }
constexpr int kSplitSmem =
    1024 + (ring_bytes(kSplitStages) > kWarpCombineBytes ? ring_bytes(kSplitStages) : kWarpCombineBytes);
static_assert(ring_bytes(kFusedStages) >= kWarpCombineBytes, "the ring doubles as the warp-combine buffer");
// the summary staging tile must hold at least 8 pages of all 128 channels (Kmax + Kmin)
static_assert(ring_bytes(kFusedStages) >= 2 * 128 * 8 * 2, "staging tile too small");

// NB: capacity of the per-sequence k1 / k2 arrays.  The fused step launches with a
// 16-entry copy when the batch allows: a 2 KB smaller parameter block measured 0.25 us
// off each launch at batch 1 on GB300.
template <int NB>
struct HsaParamsT {
  CUtensorMap tmk;         // k_pages as [num_phys*Hkv*P rows][128] bf16, 16x64 boxes, 128-B swizzle
  CUtensorMap tmv;         // v_pages, same
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
  int B, Hkv, Hq, G, P, max_pages, num_phys, nsplit, cluster, region_bytes;
  uint32_t c_mag;  // ceil(2^32 / cluster) for cluster > 1 (x / cluster as a multiply-high)
  int tok_stride;          // row stride of sigma / selp on the token path (max_pages * P)
  float scale_log2;
  int32_t k1[NB];
  int32_t k2[NB];
};
using HsaParams = HsaParamsT<RKV_MAX_BATCH>;
using HsaParamsSmall = HsaParamsT<16>;

// Current length of sequence b, clamped to the cache capacity (flagging overflow).
template <class Params>
__device__ __forceinline__ int seq_length(const Params& p, int b) {
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
  alignas(16) uint32_t ahi[128];  // rank keys: fp32 bits, or the high words of fp64 scores
  uint32_t alo[128];              // low words of the fp64 scores (fp64 path only)
  int chan[128];
  alignas(16) float qpos[128];
  alignas(16) float qneg[128];
  int warp_cnt[8];
};

// Top-k1 channels of a_i = sum_h |q_h,i| (ties: lower channel), ascending, with the
// per-channel sums of the positive and negative parts of q over the group.
// The scores are ranked exactly.  A sum of <= 8 bf16 magnitudes is usually exact in
// fp32 (each addition is checked: with x >= y >= 0, x + y is exact iff
// (x + y) - x == y); then the fp32 bit patterns rank like the exact sums.  Otherwise
// the block sums in fp64 (as the oracle does) and ranks on the fp64 bit patterns,
// high words first.  Every thread of a block of >= 128 threads calls this after
// filling qf[G][128].  on_chosen(pos, channel) runs in the thread of each chosen
// channel as soon as its place pos in the ascending list is known.
struct NoChosenHook {
  __device__ void operator()(int, int) const {}
};
template <class OnChosen = NoChosenHook>
__device__ void select_channels(const float (*qf)[128], ChanSmem& cs, int G, int k1, OnChosen on_chosen = {}) {
  const int tid = threadIdx.x;
  __syncthreads();
  float sf = 0.f;
  bool exact = true;
  if (tid < 128) {
    for (int h = 0; h < G; ++h) {
      const float x = fabsf(qf[h][tid]);
      const float big = fmaxf(sf, x), small = fminf(sf, x);
      const float sum = big + small;
      exact &= (sum - big) == small;
      sf = sum;
    }
  }
  const bool fast = __syncthreads_and(exact);
  uint32_t key = 0, lo = 0;
  if (tid < 128) {
    if (fast) {
      key = __float_as_uint(sf) + 1u;  // +1: never 0, so key - 1 below cannot wrap
    } else {
      double s = 0.0;
      for (int h = 0; h < G; ++h) s += fabs((double)qf[h][tid]);
      const unsigned long long u = (unsigned long long)__double_as_longlong(s);
      key = (uint32_t)(u >> 32);
      lo = (uint32_t)u;
      cs.alo[tid] = lo;
    }
    cs.ahi[tid] = key;
  }
  __syncthreads();
  bool sel = false;
  unsigned bal = 0;
  if (tid < 128) {
    const uint4* h4 = reinterpret_cast<const uint4*>(cs.ahi);
    const int mine = tid >> 2;
    int rank;
    if (fast) {
      // rank = #(j < tid: key_j >= key) + #(j > tid: key_j > key); a group of four
      // wholly below this channel compares against key - 1
      int r0 = 0, r1 = 0;
#pragma unroll 4  // runs once per CTA: a short body fetches fewer cold instructions
      for (int j4 = 0; j4 < 32; ++j4) {
        const uint4 u = h4[j4];
        const uint32_t t = j4 < mine ? key - 1u : key;
        r0 += (u.x > t) + (u.y > t);
        r1 += (u.z > t) + (u.w > t);
      }
      // equal keys below this channel in its own group of four (no divergent loop)
      const uint4 own = h4[mine];
      const int q = tid & 3;
      rank = r0 + r1 + (int)((q > 0) & (own.x == key)) + (int)((q > 1) & (own.y == key)) +
             (int)((q > 2) & (own.z == key));
    } else {
      int g0 = 0, g1 = 0, e0 = 0, e1 = 0;
#pragma unroll 8
      for (int j4 = 0; j4 < 32; ++j4) {
        const uint4 u = h4[j4];
        g0 += (u.x > key) + (u.y > key);
        g1 += (u.z > key) + (u.w > key);
        e0 += (u.x == key) + (u.y == key);
        e1 += (u.z == key) + (u.w == key);
      }
      rank = g0 + g1;
      if (e0 + e1 > 1) {  // another channel has the same high word: the low words decide
        const uint4* l4 = reinterpret_cast<const uint4*>(cs.alo);
        for (int j4 = 0; j4 < 32; ++j4) {
          const uint4 u = h4[j4], l = l4[j4];
          const uint32_t hv[4] = {u.x, u.y, u.z, u.w}, lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            if (hv[e] == key && j != tid) rank += (lv[e] > lo) | ((lv[e] == lo) & (j < tid));
          }
        }
      }
    }
    sel = rank < k1;
    bal = __ballot_sync(0xffffffffu, sel);
    if ((tid & 31) == 0) cs.warp_cnt[tid >> 5] = __popc(bal);
  }
  __syncthreads();
  if (tid < 128) {  // every thread computes; only the chosen channels store (predicated)
    const int w = tid >> 5;
    int pos = __popc(bal & ((1u << (tid & 31)) - 1u));
    pos += (w > 0 ? cs.warp_cnt[0] : 0) + (w > 1 ? cs.warp_cnt[1] : 0) + (w > 2 ? cs.warp_cnt[2] : 0);
    float sp = 0.f, sn = 0.f;
    for (int h = 0; h < G; ++h) {
      const float x = qf[h][tid];
      sp += fmaxf(x, 0.f);
      sn += fminf(x, 0.f);
    }
    if (sel) {
      on_chosen(pos, tid);  // the caller may start copying this channel's rows now
      cs.chan[pos] = tid;
      cs.qpos[pos] = sp;
      cs.qneg[pos] = sn;
    }
    if (tid >= k1) {  // zero past the chosen channels, so four sums load as one float4
      cs.qpos[tid] = 0.f;
      cs.qneg[tid] = 0.f;
    }
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

// Shared-memory address of 16-byte piece `piece` (channels 8*piece .. 8*piece+7) of
// token row `row` in a TMA-written K or V block: two 16 x 64 boxes (channels 0-63,
// 64-127) of 128-byte rows, each 16-byte piece XOR-ed with row % 8 (128-B swizzle;
// the block is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int piece) {
  return base + (piece >> 3) * kHalfBytes + row * 128 + ((((piece & 7) ^ (row & 7))) << 4);
}

// Barriers of one CTA's attention ring.
template <int STAGES>
struct AttnSmem {
  uint64_t bars[kAtWarps][STAGES];
  int tstart[kAtWarps][STAGES];
};

// A CTA's merged softmax state per head (unnormalised), left in its ring.
struct CtaPart {
  float M[8], L[8];
  float O[8][128];
};
constexpr int kCtaPartOffset = (kWarpCombineBytes + 255) & ~255;
static_assert(kCtaPartOffset + (int)sizeof(CtaPart) <= ring_bytes(kFusedStages), "ring too small for the partials");
static_assert((int)sizeof(TopkSmem<kThreads>) <= ring_bytes(kFusedStages), "ring too small for the top-k scratch");

// Attention of one CTA (4 warps) over items [it0, it1) of the unit's selected pages
// `sel` (ascending page ids; item i = chunk i % cpp of page sel[i / cpp]); `ptab` is
// the sequence's page-table row.  When new_pos >= 0, token new_pos is taken from
// new_kv (shared memory: its 128 K then 128 V bf16 values) instead of its cache slot,
// which may still be being written.  Leaves the CTA's merged state in the returned
// CtaPart (inside `ring`, ring_bytes(STAGES) of 1024-aligned shared memory) and sets
// *timed_out when a bounded wait ran out.
// kTok (token selection): n selected tokens, item i being tokens 16 i .. 16 i + 15;
// sel[j] is token j's row in the K/V pools (-1: zero-filled and masked), gathered row
// by row with 16-byte cp.async into the same swizzled stage layout the tiled TMA
// loads produce (rows past n are zero-filled too).
// The tiled TMA loads of chunk `chunk` of selected page `page` (of NP) into stage s of
// warp w's ring; one thread calls this.  A page id outside [0, NP) or a page-table
// entry outside the pool is flagged and its chunk masked (t0 past every token).
template <int STAGES, class Params>
__device__ __forceinline__ void load_chunk(const Params& p, AttnSmem<STAGES>& a, uint8_t* ring, int w, int s,
                                           int page, int chunk, int NP, const int32_t* ptab, int g) {
  const int P = p.P;
  const bool page_ok = page >= 0 && page < NP;  // always true for the select's output
  page = page_ok ? page : 0;
  int phys = ptab[page];
  int t0 = page * P + chunk * kChunkTok;
  if (!page_ok || phys < 0 || phys >= p.num_phys) {
    flag_error(p.err, RKV_DEVERR_PAGE_ID);
    phys = 0;
    t0 = INT_MAX / 2;  // every token of this chunk is masked
  }
  const int y = (phys * p.Hkv + g) * P + chunk * kChunkTok;
  a.tstart[w][s] = t0;
  uint8_t* st = ring + (w * STAGES + s) * kStageBytes;
  mbar_arrive_expect_tx(&a.bars[w][s], kStageBytes);
  tma_load_2d(st, &p.tmk, 0, y, &a.bars[w][s]);
  tma_load_2d(st + kHalfBytes, &p.tmk, 64, y, &a.bars[w][s]);
  tma_load_2d(st + 2 * kHalfBytes, &p.tmv, 0, y, &a.bars[w][s]);
  tma_load_2d(st + 3 * kHalfBytes, &p.tmv, 64, y, &a.bars[w][s]);
}

// bars_ready: the ring's barriers were initialised by the caller.  pre_issued: the
// caller already issued every warp's first STAGES chunks except warp kAtWarps - 1's
// last one.
template <int STAGES, bool kTok = false, class Params = HsaParams, int kG = 0>
__device__ CtaPart* attend_cta(const Params& p, const int32_t* sel, const int32_t* ptab, int b, int g, int n,
                               int it0, int it1, uint8_t* ring, AttnSmem<STAGES>& a, int new_pos,
                               const uint8_t* new_kv, int* timed_out_out, bool bars_ready = false,
                               bool pre_issued = false) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.P, G = kG > 0 ? kG : p.G;  // kG > 0: the group size known at compile time
  // page sizes are powers of two (16, 32 or 64, checked on the host): shifts, not divisions
  const int lg_p = __ffs(P) - 1;
  const int NP = (n + P - 1) >> lg_p;
  const int cpp = P / kChunkTok, lg_cpp = lg_p - 4;
  static_assert(kChunkTok == 16, "chunks of 16 tokens: cpp = P >> 4");
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
  if (!bars_ready && lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&a.bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int j) {
    const int s = j % STAGES;
    const int it = it0 + warp + j * kAtWarps;
    if constexpr (kTok) {
      // lanes 0-15: the 16 pieces of each token's K row; lanes 16-31: its V row
      const int base = it * kChunkTok, nv = min(kChunkTok, n - base);
      const int which = lane >> 4, piece = lane & 15;
      const rkv_bf16* pool = which ? p.v_pages : p.k_pages;
      uint8_t* half = wbuf + s * kStageBytes + which * 2 * kHalfBytes + (piece >> 3) * kHalfBytes;
#pragma unroll 4
      for (int r = 0; r < kChunkTok; ++r) {
        const int row = r < nv ? sel[base + r] : -1;
        cp_async16(half + r * 128 + (((piece & 7) ^ (r & 7)) << 4),
                   row >= 0 ? pool + (size_t)row * 128 + piece * 8 : pool, row >= 0 ? 16u : 0u);
      }
      cp_async_commit();
      if (lane == 0) a.tstart[warp][s] = n - nv;  // so that n - tstart counts the chunk's tokens
      __syncwarp();
      return;
    }
    if (lane == 0) load_chunk<STAGES>(p, a, ring, warp, s, sel[it >> lg_cpp], it & (cpp - 1), NP, ptab, g);
    __syncwarp();
  };

  float m_run = -1e30f, l_run = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int pre = min(nj, STAGES);
  for (int j = 0; j < pre; ++j)
    if (!pre_issued || (warp == kAtWarps - 1 && j == STAGES - 1)) issue(j);
  if constexpr (kTok)  // one cp.async group per ring slot, empty or not, so waits count evenly
    for (int j = pre; j < STAGES; ++j) cp_async_commit();
  int issued = pre, consumed = 0, timed_out = 0;
  const float sl = p.scale_log2;
  for (int j = 0; j < nj; ++j) {
    const int s = j % STAGES;
    if constexpr (kTok) {
      cp_async_wait<STAGES - 1>();  // this lane's pieces of chunk j have landed
      __syncwarp();                 // and so have the other lanes'
    } else if (!mbar_wait(&a.bars[warp][s], (uint32_t)((j / STAGES) & 1))) {
      flag_error(p.err, RKV_DEVERR_TIMEOUT);
      timed_out = 1;
      break;
    }
    uint8_t* kb = wbuf + s * kStageBytes;
    uint8_t* vb = kb + 2 * kHalfBytes;
    const int t0 = a.tstart[warp][s];
    const int nvalid = n - t0;
    const bool has_new = new_pos >= t0 && new_pos < t0 + kChunkTok;
    if (nvalid < kChunkTok || has_new) {
      if (nvalid < kChunkTok) {
        // rows past the end of the sequence hold stale data: zero their V rows (both
        // halves; the swizzle only permutes 16-B pieces within a 128-B row)
        const int nv = max(nvalid, 0);
        for (int w16 = lane; w16 < (kChunkTok - nv) * 16; w16 += 32) {
          const int row = nv + (w16 >> 4), piece = w16 & 15;
          *reinterpret_cast<uint4*>(vb + (piece >> 3) * kHalfBytes + row * 128 + (piece & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      if (has_new) {
        // the appended token: lanes 0-15 write its K pieces, lanes 16-31 its V pieces
        const int row = new_pos - t0, piece = lane & 15;
        uint8_t* dst = (lane < 16 ? kb : vb) + (piece >> 3) * kHalfBytes + row * 128 + (((piece & 7) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(new_kv + lane * 16);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    // The chunk's K and V fragments move to registers first, so its stage can be
    // refilled (the next chunk's copies issued) before the arithmetic: each warp then
    // keeps STAGES chunks in flight while it computes.
    const uint32_t kb32 = smem_u32(kb), vb32 = smem_u32(vb);
    uint32_t kf[4][2][4], vf[8][4];
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        ldsm_x4(kf[kk2][nt][0], kf[kk2][nt][1], kf[kk2][nt][2], kf[kk2][nt][3],
                swz(kb32, nt * 8 + (lane & 7), kk2 * 4 + (lane >> 3)));
#pragma unroll
    for (int nt2 = 0; nt2 < 8; ++nt2)
      ldsm_x4_t(vf[nt2][0], vf[nt2][1], vf[nt2][2], vf[nt2][3],
                swz(vb32, (lane & 7) + ((lane >> 3) & 1) * 8, nt2 * 2 + (lane >> 4)));
    // q.K^T for 16 tokens; two accumulators per n-tile shorten the MMA chains
    float sacc[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) sacc[nt][e][0] = sacc[nt][e][1] = sacc[nt][e][2] = sacc[nt][e][3] = 0.f;
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_16816(sacc[nt][0], qa0[2 * kk2], 0u, qa2[2 * kk2], 0u, kf[kk2][nt][0], kf[kk2][nt][1]);
        mma_16816(sacc[nt][1], qa0[2 * kk2 + 1], 0u, qa2[2 * kk2 + 1], 0u, kf[kk2][nt][2], kf[kk2][nt][3]);
      }
    }
    // every lane's V loads have returned (the XOR reads each fragment register) and
    // the K loads fed the MMAs above: the stage is free for the next chunk
    uint32_t vtouch = 0;
#pragma unroll
    for (int nt2 = 0; nt2 < 8; ++nt2) vtouch ^= vf[nt2][0] ^ vf[nt2][1] ^ vf[nt2][2] ^ vf[nt2][3];
    asm volatile("" ::"r"(vtouch));
    __syncwarp();
    if (j + STAGES < nj) {
      if constexpr (!kTok)
        if (lane == 0) fence_proxy_async_smem();  // the generic reads of the stage before the TMA rewrite
      issue(j + STAGES);
      issued = j + STAGES + 1;
    } else if constexpr (kTok) {
      cp_async_commit();
    }
    const int c0 = 2 * q4;
    const float z0 = (c0 < nvalid) ? (sacc[0][0][0] + sacc[0][1][0]) * sl : -INFINITY;
    const float z1 = (c0 + 1 < nvalid) ? (sacc[0][0][1] + sacc[0][1][1]) * sl : -INFINITY;
    const float z2 = (c0 + 8 < nvalid) ? (sacc[1][0][0] + sacc[1][1][0]) * sl : -INFINITY;
    const float z3 = (c0 + 9 < nvalid) ? (sacc[1][0][1] + sacc[1][1][1]) * sl : -INFINITY;
    float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    // one special-function instruction each (ex2.approx: a few ulps, results below
    // 2^-126 flushed to zero; -inf gives 0)
    const float alpha = ex2_approx(m_run - m_new);
    const float p0 = ex2_approx(z0 - m_new), p1 = ex2_approx(z1 - m_new);
    const float p2 = ex2_approx(z2 - m_new), p3 = ex2_approx(z3 - m_new);
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
      mma_16816(o[2 * nt2], ph0, 0u, ph2, 0u, vf[nt2][0], vf[nt2][1]);
      mma_16816(o[2 * nt2 + 1], ph0, 0u, ph2, 0u, vf[nt2][2], vf[nt2][3]);
      mma_16816(o[2 * nt2], pl0, 0u, pl2, 0u, vf[nt2][0], vf[nt2][1]);
      mma_16816(o[2 * nt2 + 1], pl0, 0u, pl2, 0u, vf[nt2][2], vf[nt2][3]);
    }
    consumed = j + 1;
  }
  if constexpr (kTok) cp_async_wait<0>();
  if (timed_out) {
    // wait (bounded) for this warp's copies still in flight before the ring is reused
    for (int j = consumed; j < issued; ++j) mbar_wait(&a.bars[warp][j % STAGES], (uint32_t)((j / STAGES) & 1));
  }
  *timed_out_out = __syncthreads_or(timed_out);

  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  float* cm = reinterpret_cast<float*>(ring);  // the ring is free now
  float* cl = cm + kAtWarps * 8;
  float* co = cl + kAtWarps * 8;
  CtaPart* part = reinterpret_cast<CtaPart*>(ring + kCtaPartOffset);
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
      const float f = ex2_approx(cm[w * 8 + h] - M);
      L += cl[w * 8 + h] * f;
      O += co[(w * 8 + h) * 128 + c] * f;
    }
    part->O[h][c] = O;
    if (c == 0) {
      part->M[h] = M;
      part->L[h] = L;
    }
  }
  __syncthreads();
  return part;
}

// ---------------------------------------------------------------------------
// Fused decode step.  grid (C, B*Hkv), cluster (C, 1, 1), 128 threads.
// Three instances (kMode), so that each launch holds only the once-per-CTA code it
// runs, which is fetched cold (on GB300 one kernel holding every path was 0.3-2.1 us
// a step slower): for launches whose every slice holds under 64 pages, all channels
// staged early and the top-k2 by counting ranks (at most 128 pages: kStepShortRank)
// or by the histogram select (kStepShortFlat); otherwise the chosen channels staged
// after the select and the histogram select (kStepLong).  Each also comes with the
// GQA group size fixed at 4 (kG = 4: 0.2-0.6 us a step faster on GB300, the loops over
// the group's heads unrolled) or read from the parameters (kG = 0).
// Dynamic shared memory (1024-aligned start):
//   region [region_bytes]: the query, then the staged summaries, then the K/V ring
//                          (STAGES x 4 warps x 8 KB) and the warp partials;
//   keys [max_pages] | sel [max_pages] | page-table row [max_pages];
//   inbox [C][ceil(G/C)][130] floats: the other CTAs' partial states of the heads
//                          this CTA finishes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory"); }

// Folds bf16 key x into one page's summaries in memory: *mx = max(*mx, x), *mn =
// min(*mn, x), as reductions (no load; nothing waits for them).  The reductions act
// on the 4-byte pair holding the entry; the other entry of the pair gets the identity
// of the operation (-inf for the max, +inf for the min) and keeps its value.
__device__ __forceinline__ void summary_fold(rkv_bf16* mx, rkv_bf16* mn, rkv_bf16 x) {
  const bool hi = (reinterpret_cast<uintptr_t>(mx) & 2u) != 0;  // mx and mn have the same offset in their rows
  const uint16_t ninf = 0xff80u, pinf = 0x7f80u;
  rkv_bf16* mx2 = reinterpret_cast<rkv_bf16*>(reinterpret_cast<uintptr_t>(mx) & ~(uintptr_t)3);
  rkv_bf16* mn2 = reinterpret_cast<rkv_bf16*>(reinterpret_cast<uintptr_t>(mn) & ~(uintptr_t)3);
  asm volatile("red.relaxed.gpu.global.max.noftz.v2.bf16 [%0], {%1, %2};\n" ::"l"(mx2), "h"(hi ? ninf : x),
               "h"(hi ? x : ninf)
               : "memory");
  asm volatile("red.relaxed.gpu.global.min.noftz.v2.bf16 [%0], {%1, %2};\n" ::"l"(mn2), "h"(hi ? pinf : x),
               "h"(hi ? x : pinf)
               : "memory");
}

template <int STAGES, class Params, int kMode, int kG>
__global__ void __launch_bounds__(kThreads, 2) hsa_step_kernel(const __grid_constant__ Params p) {
  constexpr bool kShort = kMode != kStepLong;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ ChanSmem cs;
  __shared__ AttnSmem<STAGES> as;
  __shared__ uint64_t sbar, pbar;
  __shared__ __align__(16) uint8_t new_kv[512];

  cg::cluster_group cluster = cg::this_cluster();
  const int C = p.cluster;
  const int rank = (int)cluster.block_rank();
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x;
  const int G = kG > 0 ? kG : p.G, P = p.P;
  uint8_t* ring = align1024(smem);
  uint32_t* keys = reinterpret_cast<uint32_t*>(ring + p.region_bytes);
  int32_t* sel = reinterpret_cast<int32_t*>(keys + p.max_pages);
  int32_t* ptab = sel + p.max_pages;
  float* inbox = reinterpret_cast<float*>(ptab + p.max_pages);
  const int hpc = C > 1 ? (int)__umulhi((uint32_t)(G + C - 1), p.c_mag) : G;  // heads finished per CTA
  // the query as floats, in the inbox (idle until the partial states arrive), so the
  // whole region is free for the summaries from the start
  float(*qf)[128] = reinterpret_cast<float(*)[128]>(inbox);

  // every CTA of the cluster must be running before anyone stores into its shared
  // memory: arrive now, wait just before the first remote store
  cluster_arrive_relaxed();
  // barriers of this CTA (shared memory only)
  if (tid == 0) {
    mbar_init(&sbar, 1);
    mbar_init(&pbar, 1);
    for (int w = 0; w < kAtWarps; ++w)  // the attention ring's (the top-k2 may fill it)
      for (int st = 0; st < STAGES; ++st) mbar_init(&as.bars[w][st], 1);
    fence_mbar_init();
  }
  // The launch may overlap the end of the previous kernel on the stream (programmatic
  // dependent launch): everything above touches only this CTA's shared memory; wait
  // here until that kernel has completed and its writes are visible, before the first
  // load.  Without such a launch this returns at once.  Before waiting, L2 is asked for
  // the small inputs read first (the sequence's length, the group's query, the new
  // token's K and V rows, the page-table row): a prefetch is only a hint, and L2 never
  // serves a line older than the writes of the kernel being waited for.  (On GB300,
  // without the length: -0.16 us a layer with 32 layers back to back, -0.15 us a step
  // at batch 16, -0.2 us at batch 1.)
  if (tid == 0) {
    prefetch_line_l2(p.seq_len + b);
    prefetch_l2(p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128, (uint32_t)G * 256);
    prefetch_l2(p.page_table + (size_t)b * p.max_pages, (uint32_t)p.max_pages * 4);
    if (p.k_new) {
      prefetch_l2(p.k_new + ((size_t)b * p.Hkv + g) * 128, 256u);
      prefetch_l2(p.v_new + ((size_t)b * p.Hkv + g) * 128, 256u);
    }
  }
  grid_dependency_wait();

  // 1. loads that depend on nothing: the group's query (16 bytes per thread), the new
  // token's K and V rows, the sequence length (one round trip for all of them)
  const rkv_bf16* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128;
  uint4 qv = make_uint4(0, 0, 0, 0), nkv = make_uint4(0, 0, 0, 0);
  if (tid < G * 16) qv = *reinterpret_cast<const uint4*>(qg + tid * 8);
  if (p.k_new && tid < 32)
    nkv = *reinterpret_cast<const uint4*>((tid < 16 ? p.k_new : p.v_new) + ((size_t)b * p.Hkv + g) * 128 +
                                          (tid & 15) * 8);
  // the length before this step; the append makes it n0 + 1
  const int cap = p.max_pages * P;
  int n0 = p.seq_len[b];
  bool do_append = p.k_new != nullptr;
  if (n0 < 0 || n0 + (do_append ? 1 : 0) > cap) {
    if (rank == 0 && tid == 0) flag_error(p.err, RKV_DEVERR_CAPACITY);
    n0 = n0 < 0 ? 0 : (n0 > cap ? cap : n0);
    do_append = false;
  }
  const int n = n0 + (do_append ? 1 : 0);
  const int lg_p = __ffs(P) - 1;  // page sizes are powers of two (16, 32 or 64, checked on the host)
  const int NP = (n + P - 1) >> lg_p;
  // 2. the append (rank 0, threads 0-63: channels 2t and 2t + 1) writes the token into
  // its slot and folds its key into its page's Kmax/Kmin.  Within this step every CTA
  // takes the token from new_kv, so nothing waits for these writes, and they need no
  // load: the fold is a max / min reduction in memory (the first token of a page
  // stores its key instead).  (On GB300 a barrier, even a warp's, waits for the loads
  // a thread has in flight, asynchronous copies included: loading the page's
  // summaries during the selection held rank 0, and with it the cluster, up by about
  // a microsecond.)
  const bool appender = do_append && rank == 0 && tid < 64;
  const int app_page = n0 >> lg_p;
  const size_t app_row = ((size_t)unit * 128 + 2 * tid) * p.max_pages + app_page;
  // this CTA's slice [p0, p1) of the pages (8-page aligned).  The short instance
  // (every slice under 64 pages) stages the summaries of all 128 channels right away,
  // in 16-byte cp.async pieces (Kmax rows 0-127, Kmin rows 128-255), while the query
  // arrives and the channels are chosen; the long one stages only the chosen
  // channels' rows, one bulk copy per row, after the select (on GB300: early
  // all-channel staging saved 0.5 us a step at 26 pages a slice; at 150-300 pages,
  // waiting for the chosen half saved 0.5-2.9 us).  The page-table row (needed after
  // the select) comes by bulk copy.
  // x / C by a multiply (c_mag = ceil(2^32 / C) from the host; exact for x < 2^31)
  auto div_c = [&](int x) { return C > 1 ? (int)__umulhi((uint32_t)x, p.c_mag) : x; };
  const int per = (div_c(NP + C - 1) + 7) & ~7;
  const int p0 = min(NP, rank * per), p1 = min(NP, p0 + per);
  const int slice8 = (p1 - p0 + 7) & ~7;
  // The short instance is launched only when every CTA's slice qualifies: a slice
  // never exceeds the one the launch computed from max_pages (the length is clamped to
  // the capacity above).  The long one never stages all channels.
  const bool all_ch = kShort && p1 > p0 && slice8 < 64 && 2 * 128 * slice8 * 2 <= p.region_bytes;
  if (all_ch) {
    const int cpr = slice8 >> 3;  // 16-byte pieces a row
    for (int i = tid; i < 256; i += kThreads) {
      const rkv_bf16* src = (i < 128 ? p.kmax : p.kmin) + ((size_t)unit * 128 + (i & 127)) * p.max_pages + p0;
      for (int c = 0; c < cpr; ++c) cp_async16(ring + (size_t)i * slice8 * 2 + c * 16, src + c * 8, 16u);
    }
    cp_async_commit();
  }
  const int np4 = ((NP + 3) & ~3);  // whole 16-byte groups; within the row (max_pages % 8 == 0)
  if (tid == 0) {
    if (np4 > 0) {
      mbar_arrive_expect_tx(&pbar, (uint32_t)np4 * 4);
      bulk_g2s(ptab, p.page_table + (size_t)b * p.max_pages, (uint32_t)np4 * 4, &pbar);
    } else {
      mbar_arrive_expect_tx(&pbar, 0);
    }
  }
  __syncthreads();

  // 3. query of the group and the new token's rows into shared memory
  if (tid < G * 16) {  // 8 channels per thread
    float* dst = &qf[tid >> 4][(tid & 15) * 8];
    dst[0] = bf16_lo(qv.x); dst[1] = bf16_hi(qv.x); dst[2] = bf16_lo(qv.y); dst[3] = bf16_hi(qv.y);
    dst[4] = bf16_lo(qv.z); dst[5] = bf16_hi(qv.z); dst[6] = bf16_lo(qv.w); dst[7] = bf16_hi(qv.w);
  }
  if (do_append && tid < 32) *reinterpret_cast<uint4*>(new_kv + tid * 16) = nkv;

  // 4. channels (every CTA).  The long instance copies the first tile of its slice's
  // chosen rows as each channel's place becomes known, inside the select.
  const int k1 = p.k1[b];
  const int tcap = kShort ? slice8 : (p.region_bytes / (4 * k1)) & ~7;  // pages a staged tile holds
  const int cnt0_8 = (min(tcap, p1 - p0) + 7) & ~7;
  const bool early_rows = !kShort && p1 > p0;
  if (early_rows && tid == 0) mbar_arrive_expect_tx(&sbar, (uint32_t)(2 * k1 * cnt0_8 * 2));
  select_channels(qf, cs, G, k1, [&](int pos, int ch) {
    if (early_rows) {
      const size_t row = ((size_t)unit * 128 + ch) * p.max_pages + p0;
      bulk_g2s(ring + (size_t)pos * cnt0_8 * 2, p.kmax + row, (uint32_t)cnt0_8 * 2, &sbar);
      bulk_g2s(ring + (size_t)(k1 + pos) * cnt0_8 * 2, p.kmin + row, (uint32_t)cnt0_8 * 2, &sbar);
    }
  });

  // 5. page bounds of this CTA's slice [p0, p1).  Staged rows: all 128 channels' Kmax
  // then Kmin (rows ch and 128 + ch), or the k1 chosen channels' (rows kk and k1 + kk,
  // copied per tile now, the region holding the whole slice whenever it fits).  The
  // appended token is folded into its
  // page's staged summary (a fold that the append may already have done changes
  // nothing: max and min are idempotent); then every thread bounds pages from shared
  // memory, and the scores go to every CTA's key array.
  const int lo_row0 = all_ch ? 128 : k1;  // Kmin row of chosen channel kk: lo_row0 + hi row
  rkv_bf16* stg = reinterpret_cast<rkv_bf16*>(ring);
  const int pnew = do_append ? n0 >> lg_p : -1;
  bool waited = false;
  int stile = 0;  // bulk-staged tiles so far (phase of sbar)
  for (int t0 = p0; t0 < p1; t0 += tcap) {
    const int cnt = min(tcap, p1 - t0);
    const int cnt8 = (cnt + 7) & ~7;  // t0 + cnt8 <= max_pages since both are multiples of 8
    __syncthreads();  // the previous tile is consumed
    if constexpr (kShort) {  // the one tile, staged at the start
      if (!all_ch) {  // cannot happen (see the launch); no scores rather than an overrun
        if (tid == 0) flag_error(p.err, RKV_DEVERR_CAPACITY);
        break;
      }
      cp_async_wait<0>();
    } else {
      // the chosen channels' rows, one bulk copy per row (the first tile's are on their
      // way since the channel select)
      if (t0 != p0) {
        fence_proxy_async_smem();
        if (tid == 0) mbar_arrive_expect_tx(&sbar, (uint32_t)(2 * k1 * cnt8 * 2));
        __syncthreads();
        for (int i = tid; i < 2 * k1; i += kThreads) {
          const rkv_bf16* base = i < k1 ? p.kmax : p.kmin;
          const int ch = cs.chan[i < k1 ? i : i - k1];
          bulk_g2s(ring + (size_t)i * cnt8 * 2, base + ((size_t)unit * 128 + ch) * p.max_pages + t0,
                   (uint32_t)cnt8 * 2, &sbar);
        }
      }
      if (!mbar_wait(&sbar, (uint32_t)(stile & 1))) flag_error(p.err, RKV_DEVERR_TIMEOUT);
      ++stile;
    }
    __syncthreads();
    if (pnew >= t0 && pnew < t0 + cnt) {
      const int j = pnew - t0;
      const bool first = (n0 & (P - 1)) == 0;
      const rkv_bf16* kn = reinterpret_cast<const rkv_bf16*>(new_kv);
      const int nrows = all_ch ? 128 : k1;
      for (int r = tid; r < nrows; r += kThreads) {
        const float x = bf16_f(kn[all_ch ? r : cs.chan[r]]);
        const int rh = r, rl = all_ch ? 128 + r : k1 + r;
        const float hi = first ? x : fmaxf(bf16_f(stg[rh * cnt8 + j]), x);
        const float lo = first ? x : fminf(bf16_f(stg[rl * cnt8 + j]), x);
        stg[rh * cnt8 + j] = (rkv_bf16)(__float_as_uint(hi) >> 16);
        stg[rl * cnt8 + j] = (rkv_bf16)(__float_as_uint(lo) >> 16);
      }
      __syncthreads();
    }
    if (!waited) {  // peers are running: their key arrays can take our scores
      cluster_wait();
      waited = true;
    }
    // row of chosen channel kk's Kmax: chan[kk] (all channels staged) or kk; its Kmin
    // row is lo_row0 further
    auto score = [&](auto all) {
      constexpr bool kAll = decltype(all)::value;
      for (int j = tid; j < cnt; j += kThreads) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // independent chains
        int kk = 0;
        for (; kk + 1 < k1; kk += 2) {
          const int r0 = kAll ? cs.chan[kk] : kk, r1 = kAll ? cs.chan[kk + 1] : kk + 1;
          s0 = fmaf(cs.qpos[kk], bf16_f(stg[r0 * cnt8 + j]), s0);
          s1 = fmaf(cs.qneg[kk], bf16_f(stg[(lo_row0 + r0) * cnt8 + j]), s1);
          s2 = fmaf(cs.qpos[kk + 1], bf16_f(stg[r1 * cnt8 + j]), s2);
          s3 = fmaf(cs.qneg[kk + 1], bf16_f(stg[(lo_row0 + r1) * cnt8 + j]), s3);
        }
        if (kk < k1) {
          const int r0 = kAll ? cs.chan[kk] : kk;
          s0 = fmaf(cs.qpos[kk], bf16_f(stg[r0 * cnt8 + j]), s0);
          s1 = fmaf(cs.qneg[kk], bf16_f(stg[(lo_row0 + r0) * cnt8 + j]), s1);
        }
        const uint32_t key = float_key((s0 + s2) + (s1 + s3));
        for (int r = 0; r < C; ++r) cluster.map_shared_rank(keys, r)[t0 + j] = key;
      }
    };
    // chosen-channel rows (long slices): a thread bounds two adjacent pages, reading
    // each row's two bf16 values as one 4-byte load (a warp reads 128 contiguous bytes
    // of a row) and four channels' q sums as one broadcast 16-byte load.  Measured on
    // GB300 in isolation (304 pages x 64 channels, 128 threads): 4,650 cycles against
    // 6,400 for one page per thread and 6,700 for four pages x a quarter of the
    // channels per lane; the loop is bound by instruction issue of its loads and FMAs.
    auto score_pairs = [&]() {
      const uint32_t* st2 = reinterpret_cast<const uint32_t*>(stg);
      const int rs2 = cnt8 >> 1;  // row stride in page pairs
      const int npairs = (cnt + 1) >> 1;
      const float4* qp4 = reinterpret_cast<const float4*>(cs.qpos);
      const float4* qn4 = reinterpret_cast<const float4*>(cs.qneg);
      const int k1r = (k1 + 3) & ~3;  // q sums are zero past k1; rows past k1 are clamped
      for (int jp = tid; jp < npairs; jp += kThreads) {
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll 2
        for (int kk = 0; kk < k1r; kk += 4) {
          const float4 qp = qp4[kk >> 2], qn = qn4[kk >> 2];
          const float qpa[4] = {qp.x, qp.y, qp.z, qp.w}, qna[4] = {qn.x, qn.y, qn.z, qn.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = min(kk + e, k1 - 1);
            const uint32_t mx = st2[r * rs2 + jp], mn = st2[(k1 + r) * rs2 + jp];
            a0 = fmaf(qpa[e], bf16_lo(mx), a0);
            a1 = fmaf(qpa[e], bf16_hi(mx), a1);
            b0 = fmaf(qna[e], bf16_lo(mn), b0);
            b1 = fmaf(qna[e], bf16_hi(mn), b1);
          }
        }
        const int j = 2 * jp;
        const uint32_t key0 = float_key(a0 + b0), key1 = float_key(a1 + b1);
        for (int r = 0; r < C; ++r) {
          uint32_t* kr = cluster.map_shared_rank(keys, r);
          kr[t0 + j] = key0;
          if (j + 1 < cnt) kr[t0 + j + 1] = key1;
        }
      }
    };
    if constexpr (kShort)
      score(std::true_type{});
    else
      score_pairs();
  }
  if (!waited) cluster_wait();
  fence_proxy_async_smem();  // generic accesses to the region before the attention's TMA loads
  cluster.sync();            // every CTA holds every page's key

  // the arrival count of sequence b's clusters: every CTA of this cluster has read the
  // length by now (before its second barrier), so the last cluster of b to count here
  // may advance seq_len (step 11).  Only the result waits, until the end.
  int arrivals = -1;
  if (do_append && rank == 0 && tid == 0) arrivals = atomicAdd(&p.sync[b], 1);

  // 6. top-k2: every CTA runs the same select over all keys (no exchange needed): by
  // counting each key's rank when the cache holds at most 128 pages, else the histogram
  // select written without divergent per-key branches (on GB300 it took 2.6 us over
  // 1212 keys where a form with per-key branches took 4.3 us, both with warm
  // instruction caches).  The list is ascending.  The select's scratch lives in the
  // ring's last stage (free between the scoring and the attention; that stage's warp
  // fills it with the rest of the attention's loads).  (The key array is 16-byte
  // aligned and followed by the list, the page-table row and the inbox, so the
  // select's reads up to 512 entries past NP stay inside this CTA's shared memory.)
  // After the histogram select the CTA's first ring fill is issued at once, one chunk
  // a thread, before the list's other uses.
  const int k = min(p.k2[b], NP);
  const int cpp = P >> 4;  // 16-token chunks a page
  const int warp_id = tid >> 5;
  const int items = k * cpp;
  const int ips = div_c(items + C - 1);
  const int it0 = min(items, rank * ips), it1 = min(items, it0 + ips);
  static_assert(sizeof(TopkSmem<kThreads>) <= kStageBytes, "the select's scratch fits one ring stage");
  TopkSmem<kThreads>& tks =
      *reinterpret_cast<TopkSmem<kThreads>*>(ring + (kAtWarps * STAGES - 1) * kStageBytes);
  if (!mbar_wait(&pbar, 0)) flag_error(p.err, RKV_DEVERR_TIMEOUT);  // the page-table row, for the loads
  bool pre_issued = false;
  if (k >= NP) {
    for (int i = tid; i < NP; i += kThreads) sel[i] = i;
  } else if constexpr (kMode == kStepShortRank) {  // NP <= max_pages <= kThreads
    topk_rank<kThreads, 1>(keys, NP, k, tks, sel);
  } else {
    topk_flat<kThreads>(keys, NP, k, tks, sel);
    // the first ring fill at once, lane s of warp w issuing warp w's chunk s (but the
    // last stage of the last warp: the select's scratch, written through the generic
    // proxy, is refilled only after the fence and barrier below)
    const int rel = warp_id + kAtWarps * (tid & 31);
    if ((tid & 31) < STAGES && rel < kAtWarps * STAGES - 1 && it0 + rel < it1)
      load_chunk<STAGES>(p, as, ring, warp_id, tid & 31, sel[(it0 + rel) >> (lg_p - 4)], (it0 + rel) & (cpp - 1), NP,
                         ptab, g);
    pre_issued = true;
  }
  if (rank == 0 && p.sel_channels && tid < 128) p.sel_channels[(size_t)unit * 128 + tid] = tid < k1 ? cs.chan[tid] : -1;
  __syncthreads();
  if (rank == 0 && p.sel_pages) {  // the caller's copy (CTA 0 only)
    int32_t* user_pages = p.sel_pages + (size_t)unit * p.sel_pages_stride;
    for (int i = tid; i < k; i += kThreads) user_pages[i] = sel[i];
    if (tid == 0 && k < p.sel_pages_stride) user_pages[k] = -1;
  }
  fence_proxy_async_smem();  // generic writes to the region before the attention's TMA loads
  __syncthreads();

  // the next kernel on the stream may start launching its CTAs into the slots this one
  // frees (it waits for this grid's completion before touching memory)
  grid_launch_dependents();
  // 7. attention over this CTA's share of the selected chunks
  int to = 0;
  const CtaPart* part =
      attend_cta<STAGES, false, Params, kG>(p, sel, ptab, b, g, n, it0, it1, ring, as, do_append ? n0 : -1, new_kv, &to,
                                            true, pre_issued);

  // 8. each head's partial state goes to the CTA that finishes the head (h % C), slot
  // [rank][h / C] of its inbox (h = j C + r)
  for (int j = 0, h = 0; h < G; ++j)
    for (int r = 0; r < C && h < G; ++r, ++h) {
      float* dst = cluster.map_shared_rank(inbox, r) + ((size_t)rank * hpc + j) * 130;
      dst[2 + tid] = part->O[h][tid];
      if (tid == 0) {
        dst[0] = part->M[h];
        dst[1] = part->L[h];
      }
    }

  cluster.sync();  // every inbox is filled; no shared memory is touched remotely after this

  // 9. merge this CTA's heads (h = j C + rank)
  for (int j = 0, h = rank; h < G; ++j, h += C) {
    float M = -1e30f;
    for (int r = 0; r < C; ++r) M = fmaxf(M, inbox[((size_t)r * hpc + j) * 130]);
    float L = 0.f, O = 0.f;
    for (int r = 0; r < C; ++r) {
      const float* src = inbox + ((size_t)r * hpc + j) * 130;
      const float f = ex2_approx(src[0] - M);
      L += src[1] * f;
      O += src[2 + tid] * f;
    }
    p.out[((size_t)b * p.Hq + (size_t)g * G + h) * 128 + tid] = L > 0.f ? O / L : 0.f;
  }

  // 10. the append's stores: the token's K and V into its slot (its physical page from
  // the page-table row), its key into the page's Kmax/Kmin
  if (appender) {
    const int app_phys = ptab[app_page];
    const uint32_t app_k = reinterpret_cast<const uint32_t*>(new_kv)[tid];
    const uint32_t app_v = reinterpret_cast<const uint32_t*>(new_kv)[64 + tid];
    if (app_phys >= 0 && app_phys < p.num_phys) {
      const int slot = n0 & (P - 1);
      const size_t dst = (((size_t)app_phys * p.Hkv + g) * P + slot) * 128 + 2 * tid;
      *reinterpret_cast<uint32_t*>(p.k_pages + dst) = app_k;
      *reinterpret_cast<uint32_t*>(p.v_pages + dst) = app_v;
      const rkv_bf16 k0 = (rkv_bf16)(app_k & 0xffffu), k1v = (rkv_bf16)(app_k >> 16);
      if (slot == 0) {  // a new page: its summaries are this key
        p.kmax[app_row] = k0;
        p.kmax[app_row + p.max_pages] = k1v;
        p.kmin[app_row] = k0;
        p.kmin[app_row + p.max_pages] = k1v;
      } else {
        summary_fold(p.kmax + app_row, p.kmin + app_row, k0);
        summary_fold(p.kmax + app_row + p.max_pages, p.kmin + app_row + p.max_pages, k1v);
      }
    } else {
      flag_error(p.err, RKV_DEVERR_PAGE_ID);
    }
  }
  // 11. the last cluster of sequence b to count advances seq_len (every CTA of every
  // cluster of b read it before that cluster counted); nothing in this launch reads it
  // again, and the next launch sees it
  if (arrivals == p.Hkv - 1) {
    p.sync[b] = 0;
    p.seq_len[b] = n;
  }
}

// ---------------------------------------------------------------------------
// Split path, steps 1-2: channel selection and page bounds into the workspace.
// grid (ceil(max_pages / 512), B*Hkv), 256 threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScoreThreads) hsa_score_kernel(const __grid_constant__ HsaParams p) {
  __shared__ ChanSmem cs;
  __shared__ float qf[8][128];
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x;
  const int n = seq_length(p, b);
  const int NP = (n + p.P - 1) / p.P;
  const int page0 = blockIdx.x * kScorePages;
  const bool write_ch = (blockIdx.x == 0) && (p.sel_channels != nullptr);
  if (page0 >= NP && !write_ch) return;
  const int G = p.G;
  const rkv_bf16* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128;
  for (int i = tid; i < G * 128; i += kScoreThreads) qf[i >> 7][i & 127] = bf16_f(qg[i]);
  const int k1 = p.k1[b];
  select_channels(qf, cs, G, k1);
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
  __shared__ TopkSmem<kTopkThreads> ts;
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
  topk_adaptive<kTopkThreads>(NP, k, [&](int i) { return keys[i]; }, ts, out, user);
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
  int to = 0;
  const CtaPart* part = attend_cta<kSplitStages>(p, p.selp + (size_t)unit * p.max_pages,
                                                 p.page_table + (size_t)b * p.max_pages, b, g, n, it0, it1,
                                                 align1024(smem), as, -1, nullptr, &to);
  if (to) return;
  const int c = threadIdx.x;
  for (int h = 0; h < p.G; ++h) {
    const size_t bh = (size_t)b * p.Hq + (size_t)g * p.G + h;
    if (p.nsplit == 1) {
      p.out[bh * 128 + c] = part->L[h] > 0.f ? part->O[h][c] / part->L[h] : 0.f;
    } else {
      p.part_o[(bh * p.nsplit + split) * 128 + c] = part->O[h][c];
      if (c == 0) p.part_ml[bh * p.nsplit + split] = make_float2(part->M[h], part->L[h]);
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

// ---------------------------------------------------------------------------
// Token path (SparQ-only: HSA with one-token pages).  With P = 1 a page's Kmax and
// Kmin are its one key, so the bound is the key's partial dot product over the chosen
// channels: s_t = sum_h sum_{i in S} q_h,i k_t,i = sum_{i in S} (sum_h q_h,i) k_t,i,
// read from the paged cache's key rows; the top-k2 tokens are attended.
// Step 1: channels and token scores.  grid (ceil(max tokens / 512), B*Hkv), 256
// threads; a half-warp scores a token (16 bytes of its row per lane), eight tokens
// rows in flight at a time.
// ---------------------------------------------------------------------------
constexpr int kTokScore = 512;  // tokens scored per CTA
__global__ void __launch_bounds__(kScoreThreads) sparq_score_kernel(const __grid_constant__ HsaParams p) {
  __shared__ ChanSmem cs;
  __shared__ float qf[8][128];
  __shared__ __align__(16) float qsel[128];
  __shared__ int sphys[kTokScore / 16];
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x;
  const int n = seq_length(p, b);
  const int t0 = blockIdx.x * kTokScore;
  const bool write_ch = (blockIdx.x == 0) && (p.sel_channels != nullptr);
  if (t0 >= n && !write_ch) return;
  const int G = p.G, P = p.P;
  const rkv_bf16* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128;
  for (int i = tid; i < G * 128; i += kScoreThreads) qf[i >> 7][i & 127] = bf16_f(qg[i]);
  const int k1 = p.k1[b];
  select_channels(qf, cs, G, k1);
  if (write_ch && tid < 128) p.sel_channels[(size_t)unit * 128 + tid] = tid < k1 ? cs.chan[tid] : -1;
  if (tid < 128) qsel[tid] = 0.f;
  __syncthreads();
  if (tid < k1) qsel[cs.chan[tid]] = cs.qpos[tid] + cs.qneg[tid];  // sum over the group's heads
  __syncthreads();
  const int piece = tid & 15;
  const float4 qa = reinterpret_cast<const float4*>(qsel)[2 * piece];
  const float4 qb = reinterpret_cast<const float4*>(qsel)[2 * piece + 1];
  const int t1 = min(n, t0 + kTokScore);
  // the physical pages of this CTA's tokens (t0 is page-aligned: P divides 512)
  const int npg = (t1 - t0 + P - 1) / P;
  for (int i = tid; i < npg; i += kScoreThreads) sphys[i] = p.page_table[(size_t)b * p.max_pages + t0 / P + i];
  __syncthreads();
  float* sg = p.sigma + (size_t)unit * p.tok_stride;
  constexpr int kU = 8;  // tokens per half-warp per pass: their rows are loaded back to back
  for (int tb = t0; tb < t1; tb += 16 * kU) {  // the same trip count for every lane
    uint4 u[kU];
    bool ok[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int t = tb + (tid >> 4) + 16 * j;
      const int lp = (t - t0) / P;
      const int phys = t < t1 ? sphys[lp] : -1;
      ok[j] = phys >= 0 && phys < p.num_phys;
      if (ok[j])
        u[j] = reinterpret_cast<const uint4*>(
            p.k_pages + (((size_t)phys * p.Hkv + g) * P + (t - t0 - lp * P)) * 128)[piece];
      else
        u[j] = make_uint4(0, 0, 0, 0);
      if (t < t1 && !ok[j] && piece == 0) flag_error(p.err, RKV_DEVERR_PAGE_ID);
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      float acc = fmaf(qa.x, bf16_lo(u[j].x), qa.y * bf16_hi(u[j].x));
      acc = fmaf(qa.z, bf16_lo(u[j].y), fmaf(qa.w, bf16_hi(u[j].y), acc));
      acc = fmaf(qb.x, bf16_lo(u[j].z), fmaf(qb.y, bf16_hi(u[j].z), acc));
      acc = fmaf(qb.z, bf16_lo(u[j].w), fmaf(qb.w, bf16_hi(u[j].w), acc));
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      const int t = tb + (tid >> 4) + 16 * j;
      if (t < t1 && piece == 0) sg[t] = ok[j] ? acc : -INFINITY;
    }
  }
}

// Token path with the channel-major key copy (SparQ's own layout: the keys stored
// once more along the head dimension, so scoring reads only the chosen channels;
// "RocketKV-adapted", "Where it sits -- the mechanism gap", SparQ-style channels).
// Per unit (b, g) the copy holds a [128][cap] bf16 block, cap = max_pages * P, row c
// = channel c of every position; a [units] int32 record counts the positions copied.
struct KeysT {
  rkv_bf16* kt;  // [units][128][cap]
  int32_t* len;  // [units]
  int32_t* chan; // [units][128] the chosen channels (workspace, this call)
  float* qs;     // [units][128] their sums of q over the group
};

// Step 0: the copy catches up with the cache: positions [len, n) of every unit (from
// len rounded down to 8, so every store is a whole 16-byte group; a record above n
// restarts at 0).  grid (units, kKtSplit), 256 threads; CTA y takes the 64-position
// tiles y, y + kKtSplit, ...  A tile's key rows are staged in shared memory, then each
// thread writes 8 positions of two channels as two 16-byte stores.  CTA 0 of a unit
// also chooses the unit's channels (into the workspace, for step 1).  The record is
// advanced by step 1, which runs after every CTA here has read it.
constexpr int kKtTile = 64, kKtSplit = 8;
__global__ void __launch_bounds__(256) sparq_keys_sync_kernel(const __grid_constant__ HsaParams p, KeysT kt) {
  __shared__ __align__(16) uint32_t tile[kKtTile][68];  // a position's 64 channel pairs (+4 pad words)
  __shared__ ChanSmem cs;
  __shared__ float qf[8][128];
  const int unit = blockIdx.x, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x;
  const int n = seq_length(p, b);
  if (blockIdx.y == 0) {
    const int G = p.G;
    const rkv_bf16* qg = p.q + ((size_t)b * p.Hq + (size_t)g * G) * 128;
    for (int i = tid; i < G * 128; i += 256) qf[i >> 7][i & 127] = bf16_f(qg[i]);
    const int k1 = p.k1[b];
    select_channels(qf, cs, G, k1);
    if (tid < 128) {
      if (p.sel_channels) p.sel_channels[(size_t)unit * 128 + tid] = tid < k1 ? cs.chan[tid] : -1;
      kt.chan[unit * 128 + tid] = tid < k1 ? cs.chan[tid] : 0;
      kt.qs[unit * 128 + tid] = tid < k1 ? cs.qpos[tid] + cs.qneg[tid] : 0.f;  // the group's sum of q
    }
  }
  int m = kt.len[unit];
  if (m < 0 || m > n) m = 0;
  const size_t cap = (size_t)p.max_pages * p.P;
  rkv_bf16* dst = kt.kt + (size_t)unit * 128 * cap;
  for (int t0 = (m & ~7) + blockIdx.y * kKtTile; t0 < n; t0 += kKtSplit * kKtTile) {
    for (int e = tid; e < kKtTile * 16; e += 256) {  // 16-byte pieces of the tile's key rows
      const int r = e >> 4, piece = e & 15, t = t0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < n) {
        const int phys = p.page_table[(size_t)b * p.max_pages + t / p.P];
        if (phys >= 0 && phys < p.num_phys)
          v = reinterpret_cast<const uint4*>(p.k_pages + (((size_t)phys * p.Hkv + g) * p.P + t % p.P) * 128)[piece];
        else if (piece == 0)
          flag_error(p.err, RKV_DEVERR_PAGE_ID);
      }
      *reinterpret_cast<uint4*>(&tile[r][piece * 4]) = v;
    }
    __syncthreads();
    const int ngrp = (min(kKtTile, n - t0) + 7) >> 3;
    for (int e = tid; e < 64 * ngrp; e += 256) {  // lanes take consecutive channel pairs
      const int c2 = e & 63, grp = e >> 6;
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = tile[grp * 8 + j][c2];
      uint4 lo, hi;  // channel 2 c2, channel 2 c2 + 1: positions in ascending order
      lo.x = (w[0] & 0xffffu) | (w[1] << 16);
      lo.y = (w[2] & 0xffffu) | (w[3] << 16);
      lo.z = (w[4] & 0xffffu) | (w[5] << 16);
      lo.w = (w[6] & 0xffffu) | (w[7] << 16);
      hi.x = (w[0] >> 16) | (w[1] & 0xffff0000u);
      hi.y = (w[2] >> 16) | (w[3] & 0xffff0000u);
      hi.z = (w[4] >> 16) | (w[5] & 0xffff0000u);
      hi.w = (w[6] >> 16) | (w[7] & 0xffff0000u);
      rkv_bf16* col = dst + (size_t)(2 * c2) * cap + t0 + grp * 8;
      *reinterpret_cast<uint4*>(col) = lo;
      *reinterpret_cast<uint4*>(col + cap) = hi;
    }
    __syncthreads();
  }
}

// Step 1 with the copy: s_t over the chosen channels (chosen in step 0), each one's
// row read from the copy.  grid (ceil(max tokens / 1024), units), 256 threads = 4
// channel groups x 64 threads of 2 x 8 positions (16-byte loads); the four groups'
// partial sums add in shared memory.  Group r takes the chosen channels r, r + 4, ...,
// four at a time (eight loads in flight a thread); the channels past k1 weigh 0.
// Positions at or past n read whatever the copy holds there (finite: keys or zeros)
// and are not written out; columns past the block's end are clamped into it.
constexpr int kTokScoreT = 1024;
__global__ void __launch_bounds__(kScoreThreads) sparq_score_t_kernel(const __grid_constant__ HsaParams p, KeysT kt) {
  __shared__ int chan[128];
  __shared__ float qs[128];
  __shared__ __align__(16) float part[4][kTokScoreT];
  const int unit = blockIdx.y, b = unit / p.Hkv;
  const int tid = threadIdx.x;
  const int n = seq_length(p, b);
  const int t0 = blockIdx.x * kTokScoreT;
  if (blockIdx.x == 0 && tid == 0) kt.len[unit] = n;  // every position below n is in the copy
  if (t0 >= n) return;
  const int k1 = p.k1[b];
  if (tid < 128) {
    chan[tid] = tid < k1 ? kt.chan[unit * 128 + tid] : 0;
    qs[tid] = tid < k1 ? kt.qs[unit * 128 + tid] : 0.f;
  }
  __syncthreads();
  const int cap = p.max_pages * p.P;
  const rkv_bf16* blk = kt.kt + (size_t)unit * 128 * cap;
  const int grp = tid >> 6, j = tid & 63;
  const int c0 = min(t0 + 8 * j, cap - 8), c1 = min(t0 + 512 + 8 * j, cap - 8);
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  const int k1r = (k1 + 15) & ~15;
#pragma unroll 1
  for (int kk = grp; kk < k1r; kk += 16) {
    uint4 u[4], v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const rkv_bf16* row = blk + (size_t)chan[kk + 4 * i] * cap;
      u[i] = *reinterpret_cast<const uint4*>(row + c0);
      v[i] = *reinterpret_cast<const uint4*>(row + c1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float q = qs[kk + 4 * i];
      const uint32_t w[8] = {u[i].x, u[i].y, u[i].z, u[i].w, v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[2 * e] = fmaf(q, bf16_lo(w[e]), acc[2 * e]);
        acc[2 * e + 1] = fmaf(q, bf16_hi(w[e]), acc[2 * e + 1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    part[grp][8 * j + e] = acc[e];
    part[grp][512 + 8 * j + e] = acc[8 + e];
  }
  __syncthreads();
  float* sg = p.sigma + (size_t)unit * p.tok_stride;
  for (int i = tid; i < kTokScoreT; i += kScoreThreads) {
    const int t = t0 + i;
    if (t < n) sg[t] = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
  }
}

// Token path, step 2: top-k2 tokens, ascending.  grid B*Hkv, 1024 threads, dynamic
// shared memory = the sequence's token count of keys (at most kTokMax).
constexpr int kTokMax = 32768;
__global__ void __launch_bounds__(kTopkThreads) sparq_topk_kernel(const __grid_constant__ HsaParams p) {
  extern __shared__ uint32_t keys[];
  __shared__ TopkSmem<kTopkThreads> ts;
  const int unit = blockIdx.x, b = unit / p.Hkv;
  const int tid = threadIdx.x;
  const int n = min(seq_length(p, b), kTokMax);
  const int k = min(p.k2[b], n);
  int32_t* out = p.selp + (size_t)unit * p.tok_stride;
  int32_t* user = p.sel_pages ? p.sel_pages + (size_t)unit * p.sel_pages_stride : nullptr;
  if (user && tid == 0 && k < p.sel_pages_stride) user[k] = -1;
  if (k >= n) {
    for (int i = tid; i < n; i += kTopkThreads) {
      out[i] = i;
      if (user) user[i] = i;
    }
    return;
  }
  const float* sg = p.sigma + (size_t)unit * p.tok_stride;
  for (int i = tid; i < n; i += kTopkThreads) keys[i] = float_key(sg[i]);
  __syncthreads();
  topk_adaptive<kTopkThreads>(n, k, [&](int i) { return keys[i]; }, ts, out, user);
}

// Token path, step 3: attention over a range of the selected tokens' 16-token chunks.
// grid (nsplit, B*Hkv), 128 threads.  Dynamic shared memory: the ring (1024-aligned),
// then the CTA's token rows (at most kTokRowItems chunks of 16).
constexpr int kTokRowItems = 512;
constexpr int kTokStages = 2;  // 2 CTAs an SM (3 stages fit one): at batch 16, 41 us a step against 59
constexpr int kTokAttendSmem = 1024 + ring_bytes(kTokStages) + 1024 + kTokRowItems * kChunkTok * 4;
static_assert(ring_bytes(kTokStages) >= kWarpCombineBytes, "the ring doubles as the warp-combine buffer");
static_assert(kTokMax / kChunkTok / kTokRowItems <= kMaxSplit, "the largest selection splits into few enough CTAs");
__global__ void __launch_bounds__(kThreads) sparq_attend_kernel(const __grid_constant__ HsaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ AttnSmem<kTokStages> as;
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv, split = blockIdx.x;
  const int n = min(seq_length(p, b), kTokMax);
  const int k = min(p.k2[b], n);
  const int items = (k + kChunkTok - 1) / kChunkTok;
  const int ips = (items + p.nsplit - 1) / p.nsplit;
  const int it0 = min(items, split * ips), it1 = min(items, it0 + ips);
  // this CTA's tokens as rows of the K/V pools, resolved once (the chunk loop then
  // issues its copies without waiting on the list or the page table)
  int32_t* rows = reinterpret_cast<int32_t*>(align1024(smem) + ring_bytes(kTokStages) + 1024);
  const int r0 = it0 * kChunkTok, r1 = min(k, it1 * kChunkTok);
  const int32_t* list = p.selp + (size_t)unit * p.tok_stride;
  const int32_t* prow = p.page_table + (size_t)b * p.max_pages;
  for (int i = r0 + (int)threadIdx.x; i < r1; i += kThreads) {
    const int t = list[i], page = t / p.P;
    const int phys = (t >= 0 && page < p.max_pages) ? prow[page] : -1;
    const bool ok = phys >= 0 && phys < p.num_phys;
    if (!ok) flag_error(p.err, RKV_DEVERR_PAGE_ID);
    rows[i - r0] = ok ? (phys * p.Hkv + g) * p.P + (t - page * p.P) : -1;
  }
  __syncthreads();
  int to = 0;
  const CtaPart* part = attend_cta<kTokStages, true>(p, rows - r0, nullptr, b, g, k, it0, it1, align1024(smem), as,
                                                       -1, nullptr, &to);
  const int c = threadIdx.x;
  for (int h = 0; h < p.G; ++h) {
    const size_t bh = (size_t)b * p.Hq + (size_t)g * p.G + h;
    if (p.nsplit == 1) {
      p.out[bh * 128 + c] = part->L[h] > 0.f ? part->O[h][c] / part->L[h] : 0.f;
    } else {
      p.part_o[(bh * p.nsplit + split) * 128 + c] = part->O[h][c];
      if (c == 0) p.part_ml[bh * p.nsplit + split] = make_float2(part->M[h], part->L[h]);
    }
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A [rows][128] bf16 page pool as a 2-D tensor map with 16-row x 64-channel boxes.
bool encode_pool_map(CUtensorMap* m, const rkv_bf16* base, uint64_t rows) {
  return encode_rows_map(m, base, rows, kChunkTok);
}

HsaParams make_params(const DecodeArgs& a, bool* ok) {
  const rkv_cache& c = a.cache;
  HsaParams p;
  const uint64_t rows = (uint64_t)c.num_phys_pages * c.Hkv * c.page_size;
  *ok = encode_pool_map(&p.tmk, c.k_pages, rows) && encode_pool_map(&p.tmv, c.v_pages, rows);
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
  p.tok_stride = c.max_pages * c.page_size;
  return p;
}

int max_items(const DecodeArgs& a) {
  int k2max = 1;
  for (int b = 0; b < a.cache.B; ++b) k2max = a.k2[b] > k2max ? a.k2[b] : k2max;
  return (k2max < a.cache.max_pages ? k2max : a.cache.max_pages) * (a.cache.page_size / kChunkTok);
}

// Dynamic shared memory of the fused kernel: 1024 (alignment) + region + key, list
// and page-table arrays + the partials inbox.
size_t fused_smem_bytes(int region, int max_pages) {
  return 1024 + (size_t)region + 3 * (size_t)max_pages * 4 + (size_t)(8 + kMaxCluster) * 130 * 4;
}

template <int STAGES, class Params, int kMode, int kG = 0>
int fused_blocks_per_sm(size_t smem) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(hsa_step_kernel<STAGES, Params, kMode, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         200 * 1024);
    attr = true;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, hsa_step_kernel<STAGES, Params, kMode, kG>, kThreads, smem) !=
      cudaSuccess)
    nb = 0;
  return nb;
}

// Launch of one instance (its shared-memory attribute set on first use).
template <int STAGES, class Params, int kMode, int kG>
cudaError_t launch_step(const cudaLaunchConfig_t& cfg, const Params& p) {
  fused_blocks_per_sm<STAGES, Params, kMode, kG>(cfg.dynamicSmemBytes);
  return cudaLaunchKernelEx(&cfg, hsa_step_kernel<STAGES, Params, kMode, kG>, p);
}

template <int STAGES, class Params, int kG>
cudaError_t launch_step_g(const cudaLaunchConfig_t& cfg, const Params& p, int mode) {
  if (mode == kStepShortRank) return launch_step<STAGES, Params, kStepShortRank, kG>(cfg, p);
  if (mode == kStepShortFlat) return launch_step<STAGES, Params, kStepShortFlat, kG>(cfg, p);
  return launch_step<STAGES, Params, kStepLong, kG>(cfg, p);
}

template <int STAGES, class Params>
cudaError_t launch_step_mode(const cudaLaunchConfig_t& cfg, const Params& p, int mode) {
  return p.G == 4 ? launch_step_g<STAGES, Params, 4>(cfg, p, mode) : launch_step_g<STAGES, Params, 0>(cfg, p, mode);
}

template <class Params>
cudaError_t launch_step_as(const cudaLaunchConfig_t& cfg, const Params& p, int stages, int mode) {
  return stages == 3 ? launch_step_mode<3, Params>(cfg, p, mode) : launch_step_mode<2, Params>(cfg, p, mode);
}

// The parameter block with 16-entry k1 / k2 arrays (batches of at most 16).
HsaParamsSmall small_params(const HsaParams& p) {
  HsaParamsSmall q;
  static_assert(offsetof(HsaParams, k1) == offsetof(HsaParamsSmall, k1), "the common prefix must match");
  std::memcpy(static_cast<void*>(&q), static_cast<const void*>(&p), offsetof(HsaParams, k1));
  for (int b = 0; b < 16; ++b) {
    q.k1[b] = b < p.B ? p.k1[b] : 0;
    q.k2[b] = b < p.B ? p.k2[b] : 0;
  }
  return q;
}

cudaError_t launch_fused(HsaParams& p, const DecodeArgs& a, cudaStream_t s) {
  const int units = a.cache.B * a.cache.Hkv;
  int k1max = 1;
  for (int b = 0; b < a.cache.B; ++b) k1max = a.k1[b] > k1max ? a.k1[b] : k1max;
  // The region must hold the ring, and should hold a whole slice of staged summaries.
  auto region_for = [&](int stages, int C) {
    const int per = ((a.cache.max_pages + C - 1) / C + 7) & ~7;
    int stage_bytes = 4 * k1max * per;
    stage_bytes = stage_bytes < 128 * 1024 ? stage_bytes : 128 * 1024;  // larger slices take several tiles
    int r = ring_bytes(stages) > stage_bytes ? ring_bytes(stages) : stage_bytes;
    return (r + 1023) & ~1023;
  };
  // CTAs per unit (the cluster size C, at most 8 and at most one per 4 attention
  // chunks) and ring stages: among the configurations whose CTAs all fit in one wave
  // of resident CTAs (C = 1 always qualifies), the one with the most CTAs, then the
  // fewest summary tiles per CTA, then the most stages.
  const int by_items = (max_items(a) + kAtWarps - 1) / kAtWarps;
  // the choice depends on nothing else, so the last one is kept per host thread
  struct Choice {
    int units, max_pages, k1max, by_items, dev, C, st;
    size_t smem;
  };
  static thread_local Choice last = {-1, -1, -1, -1, -1, 0, 0, 0};
  int dev = 0;
  cudaGetDevice(&dev);
  int best_C = 1, best_st = 2, best_tiles = 0;
  long best_ctas = -1;
  size_t best_smem = 0;
  const bool cached = last.units == units && last.max_pages == a.cache.max_pages && last.k1max == k1max &&
                      last.by_items == by_items && last.dev == dev;
  if (cached) {
    best_C = last.C;
    best_st = last.st;
    best_smem = last.smem;
  }
  for (int st = 3; st >= 2 && !cached; --st) {
    for (int C = 1; C <= kMaxCluster; ++C) {
      if (C > 1 && C > by_items) break;
      const int region = region_for(st, C);
      const size_t smem = fused_smem_bytes(region, a.cache.max_pages);
      const int occ = st == 3 ? fused_blocks_per_sm<3, HsaParams, kStepLong>(smem)
                              : fused_blocks_per_sm<2, HsaParams, kStepLong>(smem);
      if (occ < 1) continue;
      const long ctas = (long)units * C;
      if (C > 1 && ctas > (long)occ * num_sms()) continue;
      const int per = ((a.cache.max_pages + C - 1) / C + 7) & ~7;
      const int tcap = (region / (4 * k1max)) & ~7;
      const int tiles = tcap > 0 ? (per + tcap - 1) / tcap : 1 << 20;
      const bool better = ctas > best_ctas || (ctas == best_ctas && tiles < best_tiles);
      if (better) {
        best_C = C;
        best_st = st;
        best_tiles = tiles;
        best_ctas = ctas;
        best_smem = smem;
      }
    }
  }
  if (best_smem == 0) {
    best_C = 1;
    best_st = 2;
    best_smem = fused_smem_bytes(region_for(2, 1), a.cache.max_pages);
  }
  if (!cached) last = {units, a.cache.max_pages, k1max, by_items, dev, best_C, best_st, best_smem};
  p.cluster = best_C;
  p.c_mag = best_C > 1 ? 0xFFFFFFFFu / (uint32_t)best_C + 1u : 0u;
  p.region_bytes = region_for(best_st, best_C);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(best_C, (unsigned)units, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = best_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = best_C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the step's CTAs may be scheduled while the previous
  // kernel on the stream finishes (the kernel waits for it before any global access)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // a short instance when every slice (at most the one computed from max_pages) has
  // under 64 pages and all 128 channels' summaries of it fit the region; counting
  // ranks when no sequence can hold more than 128 pages
  const int per_max = ((a.cache.max_pages + best_C - 1) / best_C + 7) & ~7;
  const bool short_slices = per_max < 64 && 2 * 128 * per_max * 2 <= p.region_bytes;
  const int mode = !short_slices ? kStepLong : (a.cache.max_pages <= kThreads ? kStepShortRank : kStepShortFlat);
  cudaError_t e;
  launch_begin(K_HSA_STEP, s);
  if (a.cache.B <= 16)
    e = launch_step_as(cfg, small_params(p), best_st, mode);
  else
    e = launch_step_as(cfg, p, best_st, mode);
  launch_end(K_HSA_STEP, s);
  return e;
}

cudaError_t launch_split(HsaParams& p, const DecodeArgs& a, cudaStream_t s) {
  const rkv_cache& c = a.cache;
  const size_t units = (size_t)c.B * c.Hkv;
  const int items = max_items(a);
  static int occ = 0;
  if (occ == 0) {
    cudaFuncSetAttribute(hsa_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmem);
    cudaFuncSetAttribute(hsa_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, hsa_attend_kernel, kThreads, kSplitSmem) != cudaSuccess ||
        occ < 1)
      occ = 1;
  }
  // CTAs per unit: as many as fill one wave of resident CTAs, at most one per 4 chunks
  int nsplit = occ * num_sms() / (int)units;
  const int by_items = (items + kAtWarps - 1) / kAtWarps;
  nsplit = nsplit < by_items ? nsplit : by_items;
  nsplit = nsplit < 1 ? 1 : (nsplit > kMaxSplit ? kMaxSplit : nsplit);
  p.nsplit = nsplit;
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

size_t sparq_ws_bytes(int B, int Hq, int Hkv, int max_pages, int page_size) {
  const size_t units = (size_t)B * Hkv;
  const size_t tok = (size_t)max_pages * page_size;
  return align256(units * tok * 4) * 2 + align256((size_t)B * Hq * kMaxSplit * 128 * 4) +
         align256((size_t)B * Hq * kMaxSplit * 8) + units * 128 * 8;
}

int sparq_max_tokens() { return kTokMax; }

size_t sparq_keys_bytes(int B, int Hkv, int max_pages, int page_size) {
  const size_t units = (size_t)B * Hkv;
  return align256(units * 4) + units * 128 * (size_t)max_pages * page_size * 2;
}

cudaError_t launch_sparq(const DecodeArgs& a, cudaStream_t s) {
  bool ok = false;
  HsaParams p = make_params(a, &ok);  // the tensor maps are not used on this path
  const rkv_cache& c = a.cache;
  const size_t units = (size_t)c.B * c.Hkv;
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  const size_t sg = align256(units * (size_t)p.tok_stride * 4);
  p.sigma = reinterpret_cast<float*>(w);
  p.selp = reinterpret_cast<int32_t*>(w + sg);
  p.part_o = reinterpret_cast<float*>(w + 2 * sg);
  p.part_ml = reinterpret_cast<float2*>(w + 2 * sg + align256((size_t)c.B * a.Hq * kMaxSplit * 128 * 4));
  int kmax = 1;
  for (int b = 0; b < c.B; ++b) kmax = a.k2[b] > kmax ? a.k2[b] : kmax;
  kmax = kmax < p.tok_stride ? kmax : p.tok_stride;
  const int items = (kmax + kChunkTok - 1) / kChunkTok;
  // CTAs per unit: as many as fill one wave of resident CTAs (more waves each pay the
  // ring's fill and drain again), at most one per 4 chunks, and enough that no CTA
  // resolves more than kTokRowItems chunks' rows
  static int occ = 0;
  if (occ == 0) {
    cudaFuncSetAttribute(sparq_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTokAttendSmem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparq_attend_kernel, kThreads, kTokAttendSmem) !=
            cudaSuccess ||
        occ < 1)
      occ = 1;
  }
  int nsplit = occ * num_sms() / (int)units;
  const int by_items = (items + kAtWarps - 1) / kAtWarps;
  nsplit = nsplit < by_items ? nsplit : by_items;
  const int by_rows = (items + kTokRowItems - 1) / kTokRowItems;  // a CTA resolves at most 512 items' rows
  nsplit = nsplit > by_rows ? nsplit : by_rows;
  nsplit = nsplit < 1 ? 1 : (nsplit > kMaxSplit ? kMaxSplit : nsplit);
  p.nsplit = nsplit;
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(sparq_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTokAttendSmem);
    cudaFuncSetAttribute(sparq_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTokMax * 4);
    attrs = true;
  }
  const int ntok = p.tok_stride < kTokMax ? p.tok_stride : kTokMax;
  const dim3 score_grid((ntok + kTokScore - 1) / kTokScore, (unsigned)units);
  if (a.keys_t) {
    KeysT kt;
    kt.len = static_cast<int32_t*>(a.keys_t);
    kt.kt = reinterpret_cast<rkv_bf16*>(static_cast<uint8_t*>(a.keys_t) + align256(units * 4));
    uint8_t* chw = w + 2 * sg + align256((size_t)c.B * a.Hq * kMaxSplit * 128 * 4) +
                   align256((size_t)c.B * a.Hq * kMaxSplit * 8);
    kt.chan = reinterpret_cast<int32_t*>(chw);
    kt.qs = reinterpret_cast<float*>(chw + units * 128 * 4);
    launch_begin(K_SPARQ_KEYS_SYNC, s);
    sparq_keys_sync_kernel<<<dim3((unsigned)units, kKtSplit), 256, 0, s>>>(p, kt);
    launch_end(K_SPARQ_KEYS_SYNC, s);
    launch_begin(K_SPARQ_SCORE, s);
    sparq_score_t_kernel<<<dim3((ntok + kTokScoreT - 1) / kTokScoreT, (unsigned)units), kScoreThreads, 0, s>>>(p, kt);
    launch_end(K_SPARQ_SCORE, s);
  } else {
    launch_begin(K_SPARQ_SCORE, s);
    sparq_score_kernel<<<score_grid, kScoreThreads, 0, s>>>(p);
    launch_end(K_SPARQ_SCORE, s);
  }
  launch_begin(K_SPARQ_TOPK, s);
  sparq_topk_kernel<<<(unsigned)units, kTopkThreads, (size_t)ntok * 4, s>>>(p);
  launch_end(K_SPARQ_TOPK, s);
  launch_begin(K_SPARQ_ATTEND, s);
  sparq_attend_kernel<<<dim3(nsplit, (unsigned)units), kThreads, kTokAttendSmem, s>>>(p);
  launch_end(K_SPARQ_ATTEND, s);
  if (nsplit > 1) {
    launch_begin(K_HSA_COMBINE, s);
    hsa_combine_kernel<<<(unsigned)(c.B * a.Hq), 128, 0, s>>>(p);
    launch_end(K_HSA_COMBINE, s);
  }
  (void)ok;
  return cudaGetLastError();
}

bool decode_fused_ok(const rkv_cache& c) { return c.max_pages <= kFusedMaxPages; }

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  bool ok = false;
  HsaParams p = make_params(a, &ok);
  if (!ok) {
    set_last_error("cuTensorMapEncodeTiled failed for the K/V page pools");
    return cudaErrorInvalidValue;
  }
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
