// Stage 1 of RocketKV: SnapKV++ eviction at prefill.
//
// RocketKV abstract (arXiv 2502.14051): the first stage evicts input tokens
// coarsely with SnapKV++, SnapKV with an adaptive pooling size and full
// grouped-query-attention compatibility.  Research-map summary, "Approach":
// SnapKV with a large pooling kernel and GQA-group-level selection.
//
// Per (sequence b, KV head g) "unit", with R = G*w query rows (the G heads of the
// group times the w window queries, row r = head*w + j at position L-w+j):
//   snap_score<stats>   pass 1: per-row max and sum of exp of the scaled logits
//                       over the keys each row may see (causal), per split of L
//   snap_stats_combine  merge of the splits -> (M_r, 1/l_r)
//   snap_score<colsum>  pass 2: recompute the logits, S[t] = sum_r exp(z - M_r)/l_r
//                       for prefix tokens t < L-w (the group sum is the row sum)
//   snap_pool           centred max-pool of S (out-of-range positions ignored)
//   snap_select         block radix select of the top keep1-w pooled positions
//                       (value desc, position asc) + the window, ascending
//   snap_compact        gather of the survivors' K/V into the cache pages, their
//                       Kmax/Kmin summaries, seq_len = keep1
// The logits are tcgen05 MMAs (5th-generation tensor cores, bf16 in, fp32 out in
// tensor memory): each CTA scores a run of 128-key tiles of one unit, the tiles
// streamed in by TMA, with the unit's query rows resident in shared memory.  Pass 1
// puts the query rows on the TMEM lanes (one row per epilogue thread: the row's
// running max and sum stay in that thread); pass 2 swaps the operands so the keys
// are the lanes (one key per thread: its column sum over the rows is a private loop).
#include "rkv_device.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

constexpr int kTcTile = 128;                      // keys per tile (the MMA's M or N)
constexpr int kTcStages = 2;                      // K tiles in flight per CTA
constexpr int kTcThreads = 192;                   // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kTcOperandBytes = 128 * 256;        // 128 rows x 128 bf16: two 128 x 64 boxes
constexpr int kTcSmem = 1024 + kTcOperandBytes * (1 + kTcStages);
constexpr int kTcTmemCols = 256;                  // two 128-column fp32 accumulators
constexpr int kMaxSnapSplit = 256;
constexpr int kPoolTile = 2048;
constexpr int kPoolThreads = 256;
constexpr int kMaxPool = 255;
constexpr int kSelectThreads = 1024;
constexpr int kSelectStagedMax = 48 * 1024;  // prefix tokens whose keys the select stages (192 KB)

struct SnapParams {
  CUtensorMap tmk;        // k as [B*Hkv*Lmax rows][128] bf16, 128-row x 64-channel boxes, 128-B swizzle
  const rkv_bf16* q_win;
  const rkv_bf16* k;
  const rkv_bf16* v;
  int B, Hq, Hkv, G, w, R, Lmax, nsplit;
  int item_keys;          // keys per scoring CTA (a multiple of 128)
  int cgroup;             // pages per compaction CTA (1 .. 8)
  float scale_log2;
  float2* part;           // [units][nsplit][128] (m, l)
  float2* rowstat;        // [units][128] (M, 1/l)
  float* S;               // [units][Lmax]
  float* pooled;          // [units][Lmax]
  int32_t* kept;          // [units][kept_stride]
  int kept_stride;
  rkv_bf16* k_pages;
  rkv_bf16* v_pages;
  const int32_t* page_table;
  int32_t* seq_len;
  rkv_bf16* kmax;
  rkv_bf16* kmin;
  int32_t* err;
  int P, max_pages, num_phys;
  int32_t L[RKV_MAX_BATCH];
  int32_t keep1[RKV_MAX_BATCH];
  int32_t kp[RKV_MAX_BATCH];
};

// Byte offset of 16-byte piece `piece` (channels 8*piece .. +7) of row `row` in an
// operand laid out as TMA writes it: two 128-row x 64-channel boxes (channels 0-63,
// 64-127) of 128-byte rows, each piece XOR-ed with row % 8.
__device__ __forceinline__ uint32_t tc_swz(int row, int piece) {
  return (uint32_t)((piece >> 3) * (kTcOperandBytes / 2) + row * 128 + ((((piece & 7) ^ (row & 7))) << 4));
}

// ---------------------------------------------------------------------------
// Both passes.  grid (nsplit, B*Hkv), 192 threads, dynamic smem kTcSmem; CTA
// `split` scores keys [split * item_keys, ...) of its unit (pass 1: all L keys; pass 2:
// the L - w prefix keys).
//   warp 4 (one lane): TMA loads of the K tiles into a two-stage ring;
//   warp 5 (one lane): per tile, eight K=16 MMAs into accumulator (tile % 2) of TMEM;
//   warps 0-3: read the accumulator (thread = TMEM lane) and fold it.
// Barriers: full[s] (TMA -> MMA, transaction bytes), empty[s] (MMA commit -> TMA),
// tfull[d] (MMA commit -> epilogue), tempty[d] (128 epilogue arrivals -> MMA).  Every
// wait is bounded; a wait that runs out flags RKV_DEVERR_TIMEOUT, stops every role
// and the CTA drains what it issued before freeing TMEM.
// ---------------------------------------------------------------------------
template <bool kStats>
__global__ void __launch_bounds__(kTcThreads) snap_score_kernel(const __grid_constant__ SnapParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_b[kTcStages], empty_b[kTcStages], tfull_b[2], tempty_b[2];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  __shared__ float2 rs[128];  // pass 2: (M_r, 1/l_r)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv, split = blockIdx.x;
  const int L = p.L[b];
  const int col_end = kStats ? L : L - p.w;  // keys scored by this pass
  const int t_begin = split * p.item_keys;
  const int t_end = min(col_end, t_begin + p.item_keys);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kTcTile - 1) / kTcTile : 0;
  if (ntiles == 0) {
    if (kStats && tid < 128) p.part[((size_t)unit * p.nsplit + split) * 128 + tid] = make_float2(-1e30f, 0.f);
    return;
  }
  uint8_t* qs = align1024(smem);
  uint8_t* ks = qs + kTcOperandBytes;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&tfull_b[d], 1);
      mbar_init(&tempty_b[d], 128);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&tmem_base, kTcTmemCols);
    tmem_relinquish();
  }
  // the unit's query rows (row r = head * w + j), zero from row R on
  for (int e = tid; e < 128 * 16; e += kTcThreads) {
    const int r = e >> 4, piece = e & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < p.R)
      v = *reinterpret_cast<const uint4*>(
          p.q_win + (((size_t)b * p.Hq + (size_t)g * p.G + r / p.w) * p.w + r % p.w) * 128 + piece * 8);
    *reinterpret_cast<uint4*>(qs + tc_swz(r, piece)) = v;
  }
  if (!kStats)
    for (int r = tid; r < 128; r += kTcThreads) rs[r] = p.rowstat[(size_t)unit * 128 + r];
  fence_proxy_async_smem();  // the generic writes of Q, before the MMAs read it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  int issued = 0, committed = -1;  // TMA tiles issued (warp 4); last tile committed (warp 5)

  if (warp == 4) {
    if (lane == 0) {
      const int row0 = unit * p.Lmax + t_begin;  // rows past the unit are masked, past the array zero
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kTcStages;
        if (i >= kTcStages && !mbar_wait(&empty_b[s], (uint32_t)((i / kTcStages - 1) & 1))) {
          flag_error(p.err, RKV_DEVERR_TIMEOUT);
          abort_flag = 1;
        }
        if (abort_flag) break;
        uint8_t* st = ks + s * kTcOperandBytes;
        mbar_arrive_expect_tx(&full_b[s], kTcOperandBytes);
        tma_load_2d(st, &p.tmk, 0, row0 + i * kTcTile, &full_b[s]);
        tma_load_2d(st + kTcOperandBytes / 2, &p.tmk, 64, row0 + i * kTcTile, &full_b[s]);
        issued = i + 1;
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t q32 = smem_u32(qs), k32 = smem_u32(ks);
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kTcStages, d = i & 1;
        bool ok = mbar_wait(&full_b[s], (uint32_t)((i / kTcStages) & 1));
        if (ok && i >= 2) ok = mbar_wait(&tempty_b[d], (uint32_t)(((i >> 1) - 1) & 1));
        if (!ok) {
          flag_error(p.err, RKV_DEVERR_TIMEOUT);
          abort_flag = 1;
        }
        if (abort_flag) break;
        tc_fence_after();
        const uint32_t kt = k32 + s * kTcOperandBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kTcOperandBytes / 2) + (kk & 3) * 32;
          const uint64_t qd = sw128_kmajor_desc(q32 + off), kd = sw128_kmajor_desc(kt + off);
          tc_mma_bf16(tmem + d * 128, kStats ? qd : kd, kStats ? kd : qd, idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(&empty_b[s]);
        tc_commit(&tfull_b[d]);
        committed = i;
      }
      // the last tile's stage release lands before the CTA may exit
      if (committed >= 0 && !abort_flag)
        mbar_wait(&empty_b[committed % kTcStages], (uint32_t)((committed / kTcStages) & 1));
    }
  } else {
    // epilogue: thread tid owns TMEM lane tid (pass 1: query row tid; pass 2: key t0 + tid)
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl = p.scale_log2;
    float m_run = -1e30f, l_run = 0.f;
    const int lim = (kStats && tid < p.R) ? L - p.w + tid % p.w : -1;  // last key row tid sees
    for (int i = 0; i < ntiles; ++i) {
      const int d = i & 1;
      const bool late = !mbar_wait(&tfull_b[d], (uint32_t)((i >> 1) & 1));
      if (late) {
        flag_error(p.err, RKV_DEVERR_TIMEOUT);
        abort_flag = 1;
      }
      if (__any_sync(0xffffffffu, late || abort_flag)) break;  // warp-uniform: the TMEM loads are .aligned
      tc_fence_after();
      const int t0 = t_begin + i * kTcTile;
      if (kStats) {
        const int vis = min(t_end, lim + 1) - t0;  // keys of this tile the row sees: [0, vis)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tc_ld32_wait(lane_addr + d * 128 + c * 32, v);
          float z[32];
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            z[j] = (c * 32 + j < vis) ? __uint_as_float(v[j]) * sl : -INFINITY;
            mx = fmaxf(mx, z[j]);
          }
          const float m_new = fmaxf(m_run, mx);
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            s0 += exp2f(z[j] - m_new);
            s1 += exp2f(z[j + 1] - m_new);
          }
          l_run = l_run * exp2f(m_run - m_new) + (s0 + s1);
          m_run = m_new;
        }
      } else {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4 && c * 32 < p.R; ++c) {
          uint32_t v[32];
          tc_ld32_wait(lane_addr + d * 128 + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 a0 = rs[c * 32 + j], a1 = rs[c * 32 + j + 1];
            s0 = fmaf(exp2f(__uint_as_float(v[j]) * sl - a0.x), a0.y, s0);
            s1 = fmaf(exp2f(__uint_as_float(v[j + 1]) * sl - a1.x), a1.y, s1);
          }
        }
        const int t = t0 + tid;
        if (t < t_end) p.S[(size_t)unit * p.Lmax + t] = s0 + s1;
      }
      tc_fence_before();
      mbar_arrive(&tempty_b[d]);
    }
    if (kStats) p.part[((size_t)unit * p.nsplit + split) * 128 + tid] = make_float2(m_run, l_run);
  }

  // teardown: after a timeout, wait (bounded) for the copies and MMAs still in flight
  tc_fence_before();
  __syncthreads();
  if (abort_flag) {
    if (warp == 4 && lane == 0)
      for (int i = max(0, issued - kTcStages); i < issued; ++i)
        mbar_wait(&full_b[i % kTcStages], (uint32_t)((i / kTcStages) & 1));
    if (warp == 5 && lane == 0 && committed >= 0)
      mbar_wait(&tfull_b[committed & 1], (uint32_t)((committed >> 1) & 1));
    __syncthreads();
  }
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// Merge of the pass-1 splits.  grid B*Hkv, 128 threads (one per row).
__global__ void __launch_bounds__(128) snap_stats_combine_kernel(const __grid_constant__ SnapParams p) {
  const int unit = blockIdx.x, r = threadIdx.x;
  const float2* pp = p.part + (size_t)unit * p.nsplit * 128 + r;
  float M = -1e30f;
  for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, pp[(size_t)s * 128].x);
  float l = 0.f;
  for (int s = 0; s < p.nsplit; ++s) l += pp[(size_t)s * 128].y * exp2f(pp[(size_t)s * 128].x - M);
  // rows without keys (r >= R) get a huge M and zero weight so they add nothing
  p.rowstat[(size_t)unit * 128 + r] = (r < p.R && l > 0.f) ? make_float2(M, 1.f / l) : make_float2(1e30f, 0.f);
}

// Centred max-pool.  grid (ceil(Lmax / 2048), B*Hkv), 256 threads.
__global__ void __launch_bounds__(kPoolThreads) snap_pool_kernel(const __grid_constant__ SnapParams p) {
  __shared__ float tile[kPoolTile + kMaxPool];
  const int unit = blockIdx.y, b = unit / p.Hkv;
  const int Lp = p.L[b] - p.w;
  const int half = p.kp[b] / 2;
  const int t0 = blockIdx.x * kPoolTile;
  if (t0 >= Lp) return;
  const float* S = p.S + (size_t)unit * p.Lmax;
  for (int i = threadIdx.x; i < kPoolTile + 2 * half; i += kPoolThreads) {
    const int t = t0 - half + i;
    tile[i] = (t >= 0 && t < Lp) ? S[t] : -INFINITY;
  }
  __syncthreads();
  float* out = p.pooled + (size_t)unit * p.Lmax;
  for (int o = threadIdx.x; o < kPoolTile && t0 + o < Lp; o += kPoolThreads) {
    float m = tile[o];
    for (int j = 1; j <= 2 * half; ++j) m = fmaxf(m, tile[o + j]);
    out[t0 + o] = m;
  }
}

// Top keep1-w pooled prefix positions (value desc, position asc) + the window,
// ascending.  grid B*Hkv, 1024 threads.  kStaged: the unit's pooled scores are first
// copied into dynamic shared memory as order-preserving keys (prompts up to
// kSelectStagedMax prefix tokens); otherwise every pass of the select reads them from
// global memory (L2), lane-interleaved so that each warp load is one coalesced line.
template <bool kStaged>
__global__ void __launch_bounds__(kSelectThreads) snap_select_kernel(const __grid_constant__ SnapParams p) {
  extern __shared__ uint32_t skeys[];
  __shared__ TopkSmem<kSelectThreads> ts;
  const int unit = blockIdx.x, b = unit / p.Hkv, tid = threadIdx.x;
  const int Lp = p.L[b] - p.w;
  const int k = p.keep1[b] - p.w;
  int32_t* out = p.kept + (size_t)unit * p.kept_stride;
  for (int i = tid; i < p.w; i += kSelectThreads) out[k + i] = Lp + i;
  if (k >= Lp) {
    for (int i = tid; i < Lp; i += kSelectThreads) out[i] = i;
    return;
  }
  if (k <= 0) return;
  const float* pooled = p.pooled + (size_t)unit * p.Lmax;
  if (kStaged) {
    // eight loads in flight per thread, then the stores
    for (int i0 = tid; i0 < Lp; i0 += 8 * kSelectThreads) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j * kSelectThreads;
        v[j] = i < Lp ? pooled[i] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j * kSelectThreads;
        if (i < Lp) skeys[i] = float_key(v[j]);
      }
    }
    __syncthreads();
    topk_adaptive<kSelectThreads>(Lp, k, [&](int i) { return skeys[i]; }, ts, out, nullptr);
  } else {
    topk_strided<kSelectThreads>(Lp, k, [&](int i) { return float_key(pooled[i]); }, ts, out);
  }
}

// Survivors' K/V into the cache pages and their summaries.
// grid (ceil(max keep1 / (cgroup P)), Hkv, B), 128 threads; a CTA fills a group of
// cgroup <= 8 consecutive pages of one (sequence, KV head), P = 8 kRows.  The group's kept
// positions are read into shared memory first.  Per page, thread t moves the 16-byte
// piece t % 16 (channels 8 (t % 16) .. +7) of rows t / 16, t / 16 + 8, ... (K and V)
// and keeps their max / min, which a shuffle and a 4-warp shared-memory pass combine
// into the page's summary column of a [channel][8 pages] tile; with groups of 8, each
// channel's 8 pages then go out as one 16-byte store (the summaries are channel-major).
template <int kRows>  // rows per thread: page size / 8
__global__ void __launch_bounds__(128) snap_compact_kernel(const __grid_constant__ SnapParams p) {
  constexpr int P = 8 * kRows;
  __shared__ float red[2][4][128];
  __shared__ int32_t idx[8 * P];
  __shared__ __align__(16) uint16_t tile[2][128][8];
  const int b = blockIdx.z, g = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int unit = b * p.Hkv + g;
  const int n = p.keep1[b];
  const int pg0 = blockIdx.x * p.cgroup;
  if (blockIdx.x == 0 && g == 0 && tid == 0) p.seq_len[b] = n;
  if (pg0 * P >= n) return;
  const int npg = min(p.cgroup, (n + P - 1) / P - pg0);
  const int r_end = min(p.cgroup * P, n - pg0 * P);  // kept rows of this group
  const int32_t* kept = p.kept + (size_t)unit * p.kept_stride + (size_t)pg0 * P;
  for (int r = tid; r < r_end; r += 128) idx[r] = kept[r];
  __syncthreads();
  const int piece = tid & 15, rg = tid >> 4;
  const int L = p.L[b];
  const size_t src0 = ((size_t)b * p.Hkv + g) * p.Lmax * 128 + piece * 8;
  for (int q = 0; q < npg; ++q) {
    const int pg = pg0 + q;
    const int phys = p.page_table[(size_t)b * p.max_pages + pg];
    const bool page_ok = phys >= 0 && phys < p.num_phys;
    if (!page_ok && tid == 0) flag_error(p.err, RKV_DEVERR_PAGE_ID);
    const int cnt = min(P, n - pg * P);
    const size_t dst0 = (((size_t)(page_ok ? phys : 0) * p.Hkv + g) * P) * 128 + piece * 8;
    int t[kRows];
    uint4 kv[kRows], vv[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int r = rg + 8 * j;
      t[j] = r < cnt ? idx[q * P + r] : -1;
      const bool ok = t[j] >= 0 && t[j] < L;
      kv[j] = ok ? *reinterpret_cast<const uint4*>(p.k + src0 + (size_t)t[j] * 128) : make_uint4(0, 0, 0, 0);
      vv[j] = ok ? *reinterpret_cast<const uint4*>(p.v + src0 + (size_t)t[j] * 128) : make_uint4(0, 0, 0, 0);
    }
    float mx[8], mn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      mx[e] = -INFINITY;
      mn[e] = INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int r = rg + 8 * j;
      if (r >= cnt) continue;
      if (t[j] < 0 || t[j] >= L) {  // never expected: the select writes every position
        flag_error(p.err, RKV_DEVERR_CAPACITY);
        continue;
      }
      if (page_ok) {
        *reinterpret_cast<uint4*>(p.k_pages + dst0 + (size_t)r * 128) = kv[j];
        *reinterpret_cast<uint4*>(p.v_pages + dst0 + (size_t)r * 128) = vv[j];
      }
      const uint32_t w4[4] = {kv[j].x, kv[j].y, kv[j].z, kv[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = bf16_lo(w4[e]), x1 = bf16_hi(w4[e]);
        mx[2 * e] = fmaxf(mx[2 * e], x0);
        mx[2 * e + 1] = fmaxf(mx[2 * e + 1], x1);
        mn[2 * e] = fminf(mn[2 * e], x0);
        mn[2 * e + 1] = fminf(mn[2 * e + 1], x1);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // lanes l and l ^ 16 hold the same piece
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
      mn[e] = fminf(mn[e], __shfl_xor_sync(0xffffffffu, mn[e], 16));
    }
    if (lane < 16) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        red[0][warp][piece * 8 + e] = mx[e];
        red[1][warp][piece * 8 + e] = mn[e];
      }
    }
    __syncthreads();
    {
      const int c = tid;
      const float M = fmaxf(fmaxf(red[0][0][c], red[0][1][c]), fmaxf(red[0][2][c], red[0][3][c]));
      const float m = fminf(fminf(red[1][0][c], red[1][1][c]), fminf(red[1][2][c], red[1][3][c]));
      // the values came from bf16 bit patterns, so the top 16 bits are exact
      tile[0][c][q] = (uint16_t)(__float_as_uint(M) >> 16);
      tile[1][c][q] = (uint16_t)(__float_as_uint(m) >> 16);
    }
    __syncthreads();  // red is reused by the next page
  }
  // channel c's summaries of pages pg0 .. pg0 + npg - 1 (one 16-byte store when whole)
  const int c = tid;
  const size_t row = ((size_t)unit * 128 + c) * p.max_pages + pg0;  // 16-byte aligned when cgroup == 8
  if (npg == 8) {
    *reinterpret_cast<uint4*>(p.kmax + row) = *reinterpret_cast<const uint4*>(&tile[0][c][0]);
    *reinterpret_cast<uint4*>(p.kmin + row) = *reinterpret_cast<const uint4*>(&tile[1][c][0]);
  } else {
    for (int q = 0; q < npg; ++q) {
      p.kmax[row + q] = tile[0][c][q];
      p.kmin[row + q] = tile[1][c][q];
    }
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t prefill_ws_bytes(int B, int Hq, int Hkv, int w, int Lmax) {
  (void)Hq;
  (void)w;
  const size_t units = (size_t)B * Hkv;
  return align256(units * kMaxSnapSplit * 128 * 8) + align256(units * 128 * 8) + 2 * align256(units * Lmax * 4);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  SnapParams p;
  p.q_win = a.q_win;
  p.k = a.k;
  p.v = a.v;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.G;
  p.w = a.w;
  p.R = a.G * a.w;
  p.Lmax = a.Lmax;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const size_t units = (size_t)a.B * a.Hkv;
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  p.part = reinterpret_cast<float2*>(w);
  w += align256(units * kMaxSnapSplit * 128 * 8);
  p.rowstat = reinterpret_cast<float2*>(w);
  w += align256(units * 128 * 8);
  p.S = reinterpret_cast<float*>(w);
  w += align256(units * a.Lmax * 4);
  p.pooled = a.pooled_out ? a.pooled_out : reinterpret_cast<float*>(w);
  p.kept = a.kept_idx;
  p.kept_stride = a.kept_stride;
  p.k_pages = a.cache.k_pages;
  p.v_pages = a.cache.v_pages;
  p.page_table = a.cache.page_table;
  p.seq_len = a.cache.seq_len;
  p.kmax = a.cache.kmax;
  p.kmin = a.cache.kmin;
  p.err = a.cache.error_word;
  p.P = a.cache.page_size;
  p.max_pages = a.cache.max_pages;
  p.num_phys = a.cache.num_phys_pages;
  int Lmax_seen = 1, keep_max = 1;
  for (int b = 0; b < a.B; ++b) {
    p.L[b] = a.prompt_len[b];
    p.keep1[b] = a.keep1[b];
    p.kp[b] = a.pool_kernel[b];
    Lmax_seen = a.prompt_len[b] > Lmax_seen ? a.prompt_len[b] : Lmax_seen;
    keep_max = a.keep1[b] > keep_max ? a.keep1[b] : keep_max;
  }
  // keys per scoring CTA: 2048 (measured fastest once the grid covers the GPU), halved
  // down to 512 while there would be fewer CTAs than SMs
  p.item_keys = 2048;
  for (;;) {
    long items = 0;
    for (int b = 0; b < a.B; ++b) items += (long)a.Hkv * ((a.prompt_len[b] + p.item_keys - 1) / p.item_keys);
    if (items >= num_sms() || p.item_keys <= 512) break;
    p.item_keys /= 2;
  }
  p.nsplit = (Lmax_seen + p.item_keys - 1) / p.item_keys;
  if (p.nsplit > kMaxSnapSplit) {
    set_last_error("prompt longer than the scoring kernels' split table (524288 tokens)");
    return cudaErrorInvalidValue;
  }
  if (!encode_rows_map(&p.tmk, a.k, (uint64_t)a.B * a.Hkv * a.Lmax, kTcTile)) {
    set_last_error("cuTensorMapEncodeTiled failed for the prompt keys");
    return cudaErrorInvalidValue;
  }
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(snap_score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    cudaFuncSetAttribute(snap_score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    attrs = true;
  }
  const dim3 sgrid(p.nsplit, (unsigned)units);
  launch_begin(K_SNAP_STATS, s);
  snap_score_kernel<true><<<sgrid, kTcThreads, kTcSmem, s>>>(p);
  launch_end(K_SNAP_STATS, s);
  launch_begin(K_SNAP_STATS_COMBINE, s);
  snap_stats_combine_kernel<<<(unsigned)units, 128, 0, s>>>(p);
  launch_end(K_SNAP_STATS_COMBINE, s);
  launch_begin(K_SNAP_COLSUM, s);
  snap_score_kernel<false><<<sgrid, kTcThreads, kTcSmem, s>>>(p);
  launch_end(K_SNAP_COLSUM, s);
  launch_begin(K_SNAP_POOL, s);
  snap_pool_kernel<<<dim3((Lmax_seen + kPoolTile - 1) / kPoolTile, (unsigned)units), kPoolThreads, 0, s>>>(p);
  launch_end(K_SNAP_POOL, s);
  int Lp_max = 0;
  for (int b = 0; b < a.B; ++b) Lp_max = a.prompt_len[b] - a.w > Lp_max ? a.prompt_len[b] - a.w : Lp_max;
  static bool sel_attr = false;
  if (!sel_attr) {
    cudaFuncSetAttribute(snap_select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSelectStagedMax * 4);
    sel_attr = true;
  }
  launch_begin(K_SNAP_SELECT, s);
  if (Lp_max <= kSelectStagedMax)
    snap_select_kernel<true><<<(unsigned)units, kSelectThreads, (size_t)(Lp_max > 0 ? Lp_max : 1) * 4, s>>>(p);
  else
    snap_select_kernel<false><<<(unsigned)units, kSelectThreads, 0, s>>>(p);
  launch_end(K_SNAP_SELECT, s);
  launch_begin(K_SNAP_COMPACT, s);
  // 8 pages per CTA (whole 16-byte summary stores) while that still fills one wave of
  // resident CTAs (16 per SM), fewer pages per CTA for small caches
  p.cgroup = 8;
  while (p.cgroup > 1 && (long)((keep_max + p.cgroup * p.P - 1) / (p.cgroup * p.P)) * a.Hkv * a.B < 16L * num_sms())
    p.cgroup /= 2;
  const dim3 cgrid((keep_max + p.cgroup * p.P - 1) / (p.cgroup * p.P), a.Hkv, a.B);
  if (p.P == 16)
    snap_compact_kernel<2><<<cgrid, 128, 0, s>>>(p);
  else if (p.P == 32)
    snap_compact_kernel<4><<<cgrid, 128, 0, s>>>(p);
  else
    snap_compact_kernel<8><<<cgrid, 128, 0, s>>>(p);
  launch_end(K_SNAP_COMPACT, s);
  return cudaGetLastError();
}

}  // namespace rkv
