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
//   snap_stats_combine  merge of the splits -> lse_r = M_r + log2(l_r) (base 2)
//   snap_score<colsum>  pass 2: recompute the logits, S[t] = sum_r 2^(z - lse_r)
//                       (= sum_r exp(z - M_r) / l_r in base 2)
//                       for prefix tokens t < L-w (the group sum is the row sum)
//   snap_pool           centred max-pool of S (out-of-range positions ignored)
//   snap_select         adaptive-bin select on a thread-block cluster of the top
//                       keep1-w pooled positions (value desc, position asc) + the
//                       window, ascending
//   snap_compact        gather of the survivors' K/V into the cache pages, their
//                       Kmax/Kmin summaries, seq_len = keep1
// The logits are tcgen05 MMAs (5th-generation tensor cores, bf16 in, fp32 out in
// tensor memory): each CTA scores a run of 128-key tiles of one unit, the tiles
// streamed in by TMA, with the unit's query rows resident in shared memory.  Pass 1
// puts the query rows on the TMEM lanes (one row per epilogue thread: the row's
// running max and sum stay in that thread); pass 2 swaps the operands so the keys
// are the lanes (one key per thread: its column sum over the rows is a private loop).
#include <cooperative_groups.h>

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
constexpr int kSelectThreads = 512;
constexpr int kSelectMaxCluster = 8;
constexpr int kSelectSliceMax = 48 * 1024;  // keys a select CTA stages (192 KB of shared memory)

struct SnapParams {
  CUtensorMap tmk;        // k as [B*Hkv*Lmax rows][128] bf16, 128-row x 64-channel boxes, 128-B swizzle
  CUtensorMap tmq;        // q_win as [B*Hq*w rows][128] bf16, the same boxes
  const rkv_bf16* q_win;
  const rkv_bf16* k;
  const rkv_bf16* v;
  int B, Hq, Hkv, G, w, R, Lmax, nsplit;
  int flat;               // the scoring passes' split: 0 per unit (grid nsplit x units), 1 flat (grid N)
  int flat_ctas;          // N of pass 1 in the flat split (the combine finds each unit's slots from it)
  int item_keys;          // keys per scoring CTA (a multiple of 128)
  int cgroup;             // pages per compaction CTA (1 .. 8)
  float scale_log2;
  float2* part;           // [units][nsplit][128] (m, l)
  float* rowlse;          // [units][128] base-2 log-sum-exp of each row, +inf for rows without keys
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

// Key tiles of sequence b in a pass (pass 1: all L keys; pass 2: the L - w prefix).
template <bool kStats>
__device__ __forceinline__ int seq_tiles(const SnapParams& p, int b) {
  const int n = kStats ? p.L[b] : p.L[b] - p.w;
  return n > 0 ? (n + kTcTile - 1) / kTcTile : 0;
}

// The pass's key tiles, unit after unit (b major, then g), as one sequence; the
// cursor walks it and names each tile's unit and its index in that unit.
template <bool kStats>
struct TileCursor {
  int b, g, unit, local, ut;  // the tile's unit, its index there, the unit's tile count
  long first;                 // sequence index of the unit's first tile
  __device__ void start(const SnapParams& p, long x) {
    b = 0;
    first = 0;
    for (;;) {
      ut = seq_tiles<kStats>(p, b);
      const long n = (long)p.Hkv * ut;
      if (x - first < n || b == p.B - 1) break;
      first += n;
      ++b;
    }
    g = ut > 0 ? (int)((x - first) / ut) : 0;
    first += (long)g * ut;
    local = (int)(x - first);
    unit = b * p.Hkv + g;
  }
  __device__ void next(const SnapParams& p) {  // past the last tile it stays in the last sequence
    if (++local < ut) return;
    first += ut;
    local = 0;
    if (++g == p.Hkv) {
      g = 0;
      while (b + 1 < p.B) {
        ut = seq_tiles<kStats>(p, ++b);
        if (ut > 0) break;
      }
    }
    unit = b * p.Hkv + g;
  }
};

// In the flat split (gridDim.x = N CTAs over the T tiles of the sequence), CTA i takes
// tiles [i T / N, (i + 1) T / N); the CTA holding tile x is ceil((x + 1) N / T) - 1.
__device__ __forceinline__ int flat_cta_of(long x, long T, int N) { return (int)(((x + 1) * N - 1) / T); }

template <bool kStats>
__device__ __forceinline__ long pass_tiles_total(const SnapParams& p) {
  long T = 0;
  for (int b = 0; b < p.B; ++b) T += (long)p.Hkv * seq_tiles<kStats>(p, b);
  return T;
}

// ---------------------------------------------------------------------------
// Both passes, 192 threads, dynamic smem kTcSmem.  Split per unit (flat == 0): grid
// (nsplit, B*Hkv), CTA `split` scores tiles [split * item_keys / 128, ...) of its unit.
// Flat split (flat == 1): grid (N), CTA i scores its equal share of the pass's tiles
// taken unit after unit, so that every resident-CTA slot is used when the units do
// not divide the slots; a share may run across units (the query tile is then
// reloaded and, in pass 1, the row statistics are written per unit).  Pass 1 scores
// all L keys, pass 2 the L - w prefix keys.
//   warp 4 (one lane): TMA loads of each unit's query tile and of the K tiles into a
//                      two-stage ring;
//   warp 5 (one lane): per tile, eight K=16 MMAs into accumulator (tile % 2) of TMEM;
//   warps 0-3: read the accumulator (thread = TMEM lane) and fold it.
// Barriers: qfull (query TMA -> MMA, one phase per unit), full[s] (TMA -> MMA,
// transaction bytes), empty[s] (MMA commit -> TMA; it also tells the TMA warp that
// the query tile is free), tfull[d] (MMA commit -> epilogue), tempty[d] (128 epilogue
// arrivals -> MMA).  Every wait is bounded; a wait that runs out flags
// RKV_DEVERR_TIMEOUT, stops every role and the CTA drains what it issued before
// freeing TMEM.  The query tile is the unit's R = G w rows (row r = head * w + j) and
// then whatever follows them in q_win (zero past its end): pass 1 masks rows from R
// on, pass 2 weighs them by 2^-inf = 0.
// ---------------------------------------------------------------------------
template <bool kStats>
__global__ void __launch_bounds__(kTcThreads) snap_score_kernel(const __grid_constant__ SnapParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_b[kTcStages], empty_b[kTcStages], tfull_b[2], tempty_b[2], qfull_b;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  __shared__ __align__(16) float rs[4][128];  // pass 2: lse_r = M_r + log2(l_r) (base 2), per epilogue warp

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  // this CTA's run of tiles: ntiles from the cursor's start
  TileCursor<kStats> cur0;
  int ntiles, split = 0;
  long T = 0;
  if (p.flat) {
    T = pass_tiles_total<kStats>(p);
    const int N = gridDim.x, i = blockIdx.x;
    const long g0 = (long)i * T / N, g1 = (long)(i + 1) * T / N;
    ntiles = (int)(g1 - g0);
    if (ntiles > 0) cur0.start(p, g0);
  } else {
    const int unit = blockIdx.y, b = unit / p.Hkv;
    split = blockIdx.x;
    const int ut = seq_tiles<kStats>(p, b), per = p.item_keys / kTcTile;
    ntiles = max(0, min(per, ut - split * per));
    cur0.b = b;
    cur0.g = unit % p.Hkv;
    cur0.unit = unit;
    cur0.ut = ut;
    cur0.local = split * per;
    cur0.first = 0;  // unused: the run stays in its unit
  }
  if (ntiles == 0) {
    if (kStats && !p.flat && tid < 128)
      p.part[((size_t)blockIdx.y * p.nsplit + split) * 128 + tid] = make_float2(-1e30f, 0.f);
    return;
  }
  // pass-1 slot of this CTA's statistics for the unit whose first tile is `first`
  auto slot_of = [&](long first) { return p.flat ? blockIdx.x - flat_cta_of(first, T, gridDim.x) : split; };
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
    mbar_init(&qfull_b, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&tmem_base, kTcTmemCols);
    tmem_relinquish();
  }
  if (!kStats && warp < 4)
    for (int r = lane; r < 128; r += 32) rs[warp][r] = p.rowlse[(size_t)cur0.unit * 128 + r];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  int issued = 0, committed = -1, qissued = 0;  // K tiles issued, query tiles issued (warp 4); last tile committed (warp 5)
  // first query row of a unit in q_win ([B][Hq][w][128])
  auto qrow0 = [&](int b, int g) { return ((b * p.Hq + g * p.G) * p.w); };

  if (warp == 4) {
    if (lane == 0) {
      TileCursor<kStats> c = cur0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kTcStages;
        const bool new_unit = i == 0 || c.local == 0;
        if (i >= kTcStages && !mbar_wait(&empty_b[s], (uint32_t)((i / kTcStages - 1) & 1))) {
          flag_error(p.err, RKV_DEVERR_TIMEOUT);
          abort_flag = 1;
        }
        if (abort_flag) break;
        uint8_t* st = ks + s * kTcOperandBytes;
        const int row = c.unit * p.Lmax + c.local * kTcTile;  // rows past the unit are masked, past the array zero
        mbar_arrive_expect_tx(&full_b[s], kTcOperandBytes);
        tma_load_2d(st, &p.tmk, 0, row, &full_b[s]);
        tma_load_2d(st + kTcOperandBytes / 2, &p.tmk, 64, row, &full_b[s]);
        issued = i + 1;
        if (new_unit) {
          // the query tile is free once the previous tile's MMAs have completed
          if (i > 0 && !mbar_wait(&empty_b[(i - 1) % kTcStages], (uint32_t)(((i - 1) / kTcStages) & 1))) {
            flag_error(p.err, RKV_DEVERR_TIMEOUT);
            abort_flag = 1;
            break;
          }
          const int qr = qrow0(c.b, c.g);
          mbar_arrive_expect_tx(&qfull_b, kTcOperandBytes);
          tma_load_2d(qs, &p.tmq, 0, qr, &qfull_b);
          tma_load_2d(qs + kTcOperandBytes / 2, &p.tmq, 64, qr, &qfull_b);
          ++qissued;
        }
        c.next(p);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t q32 = smem_u32(qs), k32 = smem_u32(ks);
      TileCursor<kStats> c = cur0;
      int qseen = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kTcStages, d = i & 1;
        bool ok = true;
        if (i == 0 || c.local == 0) ok = mbar_wait(&qfull_b, (uint32_t)(qseen++ & 1));
        if (ok) ok = mbar_wait(&full_b[s], (uint32_t)((i / kTcStages) & 1));
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
        c.next(p);
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
    TileCursor<kStats> c = cur0;
    // the last key row tid sees in its unit (-1: a row past R, which sees none)
    auto last_key = [&](int b) { return (kStats && tid < p.R) ? p.L[b] - p.w + tid % p.w : -1; };
    int lim = last_key(c.b);
    for (int i = 0; i < ntiles; ++i) {
      const int d = i & 1;
      const bool late = !mbar_wait(&tfull_b[d], (uint32_t)((i >> 1) & 1));
      if (late) {
        flag_error(p.err, RKV_DEVERR_TIMEOUT);
        abort_flag = 1;
      }
      if (__any_sync(0xffffffffu, late || abort_flag)) break;  // warp-uniform: the TMEM loads are .aligned
      tc_fence_after();
      const int t0 = c.local * kTcTile;
      if (kStats) {
        const int vis = lim + 1 - t0;  // keys of this tile the row sees: [0, vis)
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tc_ld32_wait(lane_addr + d * 128 + cc * 32, v);
          float s0 = 0.f, s1 = 0.f, m_new;
          if (cc * 32 + 32 <= vis) {  // the row sees the whole chunk: no mask; sl > 0, so max(v)*sl = max(v*sl)
            float mx = __uint_as_float(v[0]);
#pragma unroll
            for (int j = 1; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(v[j]));
            m_new = fmaxf(m_run, mx * sl);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              s0 += ex2_approx(fmaf(__uint_as_float(v[j]), sl, -m_new));
              s1 += ex2_approx(fmaf(__uint_as_float(v[j + 1]), sl, -m_new));
            }
          } else {
            float z[32];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              z[j] = (cc * 32 + j < vis) ? __uint_as_float(v[j]) * sl : -INFINITY;
              mx = fmaxf(mx, z[j]);
            }
            m_new = fmaxf(m_run, mx);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              s0 += ex2_approx(z[j] - m_new);
              s1 += ex2_approx(z[j + 1] - m_new);
            }
          }
          l_run = l_run * ex2_approx(m_run - m_new) + (s0 + s1);
          m_run = m_new;
        }
      } else {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
        for (int cc = 0; cc < 4 && cc * 32 < p.R; ++cc) {
          uint32_t v[32];
          tc_ld32_wait(lane_addr + d * 128 + cc * 32, v);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {  // p = 2^(z - M_r) / l_r = 2^(z - lse_r)
            const float4 a = *reinterpret_cast<const float4*>(&rs[warp][cc * 32 + j]);
            s0 += ex2_approx(fmaf(__uint_as_float(v[j]), sl, -a.x));
            s1 += ex2_approx(fmaf(__uint_as_float(v[j + 1]), sl, -a.y));
            s0 += ex2_approx(fmaf(__uint_as_float(v[j + 2]), sl, -a.z));
            s1 += ex2_approx(fmaf(__uint_as_float(v[j + 3]), sl, -a.w));
          }
        }
        const int t = t0 + tid;
        if (t < p.L[c.b] - p.w) p.S[(size_t)c.unit * p.Lmax + t] = s0 + s1;
      }
      tc_fence_before();
      mbar_arrive(&tempty_b[d]);
      // the unit's last tile of this run: pass 1 writes the unit's row statistics;
      // pass 2 takes the next unit's row log-sum-exps (this warp's copy)
      const bool unit_done = c.local + 1 == c.ut || i + 1 == ntiles;
      if (unit_done && kStats) {
        p.part[((size_t)c.unit * p.nsplit + slot_of(c.first)) * 128 + tid] = make_float2(m_run, l_run);
        m_run = -1e30f;
        l_run = 0.f;
      }
      c.next(p);
      if (unit_done && i + 1 < ntiles) {
        if (kStats) {
          lim = last_key(c.b);
        } else {
          __syncwarp();  // every lane has read this warp's copy for the previous unit
          for (int r = lane; r < 128; r += 32) rs[warp][r] = p.rowlse[(size_t)c.unit * 128 + r];
          __syncwarp();
        }
      }
    }
  }

  // teardown: after a timeout, wait (bounded) for the copies and MMAs still in flight
  tc_fence_before();
  __syncthreads();
  if (abort_flag) {
    if (warp == 4 && lane == 0) {
      for (int i = max(0, issued - kTcStages); i < issued; ++i)
        mbar_wait(&full_b[i % kTcStages], (uint32_t)((i / kTcStages) & 1));
      if (qissued > 0) mbar_wait(&qfull_b, (uint32_t)((qissued - 1) & 1));
    }
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
  int nparts = p.nsplit;  // split per unit: every slot written
  if (p.flat) {           // the CTAs whose runs meet this unit's pass-1 tiles
    const int b = unit / p.Hkv, g = unit % p.Hkv;
    long first = 0;
    for (int bb = 0; bb < b; ++bb) first += (long)p.Hkv * seq_tiles<true>(p, bb);
    const int ut = seq_tiles<true>(p, b);
    first += (long)g * ut;
    const long T = pass_tiles_total<true>(p);
    nparts = flat_cta_of(first + ut - 1, T, p.flat_ctas) - flat_cta_of(first, T, p.flat_ctas) + 1;
  }
  float M = -1e30f;
  for (int s = 0; s < nparts; ++s) M = fmaxf(M, pp[(size_t)s * 128].x);
  float l = 0.f;
  for (int s = 0; s < nparts; ++s) l += pp[(size_t)s * 128].y * exp2f(pp[(size_t)s * 128].x - M);
  // rows without keys (r >= R) get +inf, so 2^(z - lse) = 0 and they add nothing
  p.rowlse[(size_t)unit * 128 + r] = (r < p.R && l > 0.f) ? M + log2f(l) : INFINITY;
}

// Centred max-pool.  grid (ceil(Lmax / 2048), B*Hkv), 256 threads.
// The tile and its halo are staged once; window maxima of doubling length are built
// in place by ping-pong passes (after pass j, M[i] = max of x[i .. i + 2^j)), so a
// window of kp positions is the max of two overlapping windows of 2^j <= kp: two
// reads per output after log2(kp) passes, instead of kp reads.  Max is exact, so the
// result equals the direct definition bit for bit.
__global__ void __launch_bounds__(kPoolThreads) snap_pool_kernel(const __grid_constant__ SnapParams p) {
  __shared__ float buf[2][kPoolTile + kMaxPool];
  const int unit = blockIdx.y, b = unit / p.Hkv;
  const int Lp = p.L[b] - p.w;
  const int kp = p.kp[b], half = kp / 2;
  const int t0 = blockIdx.x * kPoolTile;
  if (t0 >= Lp) return;
  const float* S = p.S + (size_t)unit * p.Lmax;
  const int n = kPoolTile + 2 * half;  // x[i] = S[t0 - half + i], -inf outside the prefix
  for (int i = threadIdx.x; i < n; i += kPoolThreads) {
    const int t = t0 - half + i;
    buf[0][i] = (t >= 0 && t < Lp) ? S[t] : -INFINITY;
  }
  int cur = 0, w = 1;
  while (2 * w <= kp) {  // windows of w -> 2w (only the entries a later read needs)
    __syncthreads();
    const float* a = buf[cur];
    float* o = buf[cur ^ 1];
    for (int i = threadIdx.x; i + 2 * w <= n; i += kPoolThreads) o[i] = fmaxf(a[i], a[i + w]);
    cur ^= 1;
    w *= 2;
  }
  __syncthreads();
  const float* M = buf[cur];
  float* out = p.pooled + (size_t)unit * p.Lmax;
  for (int o = threadIdx.x; o < kPoolTile && t0 + o < Lp; o += kPoolThreads)
    out[t0 + o] = fmaxf(M[o], M[o + kp - w]);  // [o, o + w) and [o + kp - w, o + kp)
}

// Top keep1-w pooled prefix positions (value desc, position asc) + the window,
// ascending.  One thread-block cluster of C CTAs per unit: grid (C, B*Hkv), cluster
// (C, 1, 1), 512 threads.  CTA r stages prefix positions [r per, r per + per) as
// order-preserving keys in shared memory and the select of topk_adaptive runs over
// the cluster: the key range, each round's 1024-bin histogram, the boundary
// candidates and the compaction totals are combined through distributed shared
// memory (every CTA derives the same boundary), and each CTA writes the selected
// positions of its own slice at its offset in the ascending list.
struct SelectSmem {
  uint32_t hist[kTkBins];  // this CTA's histogram (read by every CTA of the cluster)
  uint32_t lo, hi;         // this CTA's key range
  int cnt1, cnt2;          // this CTA's taken / boundary-by-index counts
  int ncand;               // rank 0: candidates gathered from the cluster
  int cand[kTkCand];
  uint32_t ckey[kTkCand];
  uint32_t T;              // the boundary pair, written into every CTA by rank 0
  int tI;
  uint32_t wlo[kSelectThreads / 32], whi[kSelectThreads / 32];
  int wa[kSelectThreads / 32], wb[kSelectThreads / 32];
  int bstar, need, nb;
};

__global__ void __launch_bounds__(kSelectThreads) snap_select_kernel(const __grid_constant__ SnapParams p) {
  extern __shared__ uint32_t skeys[];
  __shared__ SelectSmem ss;
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int NT = kSelectThreads, NW = NT / 32, BPT = kTkBins / NT;
  const int C = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int unit = blockIdx.y, b = unit / p.Hkv, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Lp = p.L[b] - p.w;
  const int k = p.keep1[b] - p.w;
  int32_t* out = p.kept + (size_t)unit * p.kept_stride;
  // the same branch in every CTA of the cluster: no cluster barrier is skipped by some
  if (k >= Lp || k <= 0) {
    if (rank == 0)
      for (int i = tid; i < p.w; i += NT) out[k + i] = Lp + i;
    if (k >= Lp)
      for (int i = rank * NT + tid; i < Lp; i += C * NT) out[i] = i;
    return;
  }
  if (rank == 0)
    for (int i = tid; i < p.w; i += NT) out[k + i] = Lp + i;
  const int per = (Lp + C - 1) / C;
  const int s0 = min(Lp, rank * per), s1 = min(Lp, s0 + per), nl = s1 - s0;
  const float* pooled = p.pooled + (size_t)unit * p.Lmax + s0;
  // stage this slice's keys (eight loads in flight per thread) and its range
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i0 = tid; i0 < nl; i0 += 8 * NT) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = i0 + j * NT < nl ? pooled[i0 + j * NT] : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (i0 + j * NT < nl) {
        const uint32_t u = float_key(v[j]);
        skeys[i0 + j * NT] = u;
        lo = min(lo, u);
        hi = max(hi, u);
      }
  }
  lo = __reduce_min_sync(FULL, lo);
  hi = __reduce_max_sync(FULL, hi);
  if (lane == 0) {
    ss.wlo[warp] = lo;
    ss.whi[warp] = hi;
  }
  if (tid == 0) ss.ncand = 0;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < NW; ++w) {
      lo = min(lo, ss.wlo[w]);
      hi = max(hi, ss.whi[w]);
    }
    ss.lo = lo;
    ss.hi = hi;
  }
  cluster.sync();
  {
    uint32_t rl[kSelectMaxCluster], rh[kSelectMaxCluster];
#pragma unroll
    for (int r = 0; r < kSelectMaxCluster; ++r) {
      rl[r] = r < C ? cluster.map_shared_rank(&ss, r)->lo : 0xffffffffu;
      rh[r] = r < C ? cluster.map_shared_rank(&ss, r)->hi : 0u;
    }
    lo = 0xffffffffu;
    hi = 0u;
#pragma unroll
    for (int r = 0; r < kSelectMaxCluster; ++r) {
      lo = min(lo, rl[r]);
      hi = max(hi, rh[r]);
    }
  }
  // thread t owns the contiguous local keys [t seg, t seg + seg), seg odd
  const int seg = ((nl + NT - 1) / NT) | 1;
  const int t0 = min(nl, tid * seg), t1 = min(nl, t0 + seg);

  int need = k, nin = Lp;
  while (nin > kTkCand && lo != hi) {
    const uint32_t range = hi - lo;
    const int shift = range < (uint32_t)kTkBins ? 0 : (32 - __clz(range)) - 10;
    for (int i = tid; i < kTkBins; i += NT) ss.hist[i] = 0u;
    __syncthreads();
    int run_bin = -1, run = 0;
    for (int i = t0; i < t1; ++i) {
      const uint32_t u = skeys[i];
      const int bin = (u >= lo && u <= hi) ? (int)((u - lo) >> shift) : -1;
      if (bin != run_bin) {
        if (run_bin >= 0) atomicAdd(&ss.hist[run_bin], (uint32_t)run);
        run_bin = bin;
        run = 0;
      }
      ++run;
    }
    if (run_bin >= 0) atomicAdd(&ss.hist[run_bin], (uint32_t)run);
    cluster.sync();  // every CTA's histogram is complete
    uint32_t c[BPT];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      uint32_t v[kSelectMaxCluster];  // every CTA's count of the bin, loads in flight together
#pragma unroll
      for (int r = 0; r < kSelectMaxCluster; ++r) v[r] = r < C ? cluster.map_shared_rank(ss.hist, r)[tid * BPT + j] : 0u;
      c[j] = 0;
#pragma unroll
      for (int r = 0; r < kSelectMaxCluster; ++r) c[j] += v[r];
      sum += (int)c[j];
    }
    int incl = sum;  // over the lanes >= this one
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(FULL, incl, o);
      if (lane + o < 32) incl += y;
    }
    if (lane == 0) ss.wa[warp] = incl;
    __syncthreads();
    int above = incl - sum;
    for (int w = warp + 1; w < NW; ++w) above += ss.wa[w];
    if (above < need && above + sum >= need) {
      int acc = above;
#pragma unroll
      for (int j = BPT - 1; j >= 0; --j) {
        if (acc + (int)c[j] >= need) {
          ss.bstar = tid * BPT + j;
          ss.need = need - acc;
          ss.nb = (int)c[j];
          break;
        }
        acc += (int)c[j];
      }
    }
    cluster.sync();  // every CTA has read every histogram (they are cleared next round)
    const uint32_t nlo = lo + ((uint32_t)ss.bstar << shift);
    hi = shift == 0 ? nlo : min(hi, nlo + ((1u << shift) - 1u));
    lo = nlo;
    need = ss.need;
    nin = ss.nb;
  }

  const bool all_in = need == nin;
  const bool by_index = !all_in && nin > kTkCand;  // then lo == hi
  if (!by_index && !all_in) {
    // candidates into rank 0's list, ranked there; (T, t) sent to every CTA
    SelectSmem* r0 = cluster.map_shared_rank(&ss, 0);
    for (int i = t0; i < t1; ++i) {
      const uint32_t u = skeys[i];
      if (u >= lo && u <= hi) {
        const int slot = atomicAdd(&r0->ncand, 1);
        if (slot < kTkCand) {
          r0->cand[slot] = s0 + i;
          r0->ckey[slot] = u;
        }
      }
    }
    cluster.sync();
    if (rank == 0 && warp == 0) {
      const int nc = min(ss.ncand, kTkCand);
      const int ci = lane < nc ? ss.cand[lane] : 0;
      const uint32_t cu = lane < nc ? ss.ckey[lane] : 0u;
      int r = 0;
#pragma unroll
      for (int m = 0; m < 32; ++m) {
        const uint32_t a2 = __shfl_sync(FULL, cu, m);
        const int cm = __shfl_sync(FULL, ci, m);
        r += (m < nc) & ((a2 > cu) | ((a2 == cu) & (cm < ci)));
      }
      if (lane < nc && r == need - 1)
        for (int q = 0; q < C; ++q) {
          SelectSmem* o = cluster.map_shared_rank(&ss, q);
          o->T = cu;
          o->tI = ci;
        }
    }
    cluster.sync();
  }
  const uint32_t T = (by_index || all_in) ? lo : ss.T;
  const int tI = (by_index || all_in) ? Lp : ss.tI;
  auto pick = [&](int i) -> int {  // i: local index
    const uint32_t u = skeys[i];
    if (u > hi) return 1;
    if (u < lo) return 0;
    if (by_index) return 2;
    return (u > T || (u == T && s0 + i <= tI)) ? 1 : 0;
  };
  // compaction: thread counts, block scan, cluster totals, then the writes
  int c1 = 0, c2 = 0;
  for (int i = t0; i < t1; ++i) {
    const int t = pick(i);
    c1 += t == 1;
    c2 += t == 2;
  }
  int x1 = c1, x2 = c2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y1 = __shfl_up_sync(FULL, x1, o), y2 = __shfl_up_sync(FULL, x2, o);
    if (lane >= o) {
      x1 += y1;
      x2 += y2;
    }
  }
  if (lane == 31) {
    ss.wa[warp] = x1;
    ss.wb[warp] = x2;
  }
  __syncthreads();
  int base = x1 - c1, bseen = x2 - c2;
  for (int w = 0; w < warp; ++w) {
    base += ss.wa[w];
    bseen += ss.wb[w];
  }
  if (tid == NT - 1) {
    ss.cnt1 = base + c1;
    ss.cnt2 = bseen + c2;
  }
  cluster.sync();  // every CTA's totals are in place
  {
    int a1[kSelectMaxCluster], a2[kSelectMaxCluster];
#pragma unroll
    for (int r = 0; r < kSelectMaxCluster; ++r) {
      a1[r] = r < rank ? cluster.map_shared_rank(&ss, r)->cnt1 : 0;
      a2[r] = r < rank ? cluster.map_shared_rank(&ss, r)->cnt2 : 0;
    }
#pragma unroll
    for (int r = 0; r < kSelectMaxCluster; ++r) {
      base += a1[r];
      bseen += a2[r];
    }
  }
  cluster.sync();  // no CTA leaves while another still reads its shared memory
  int o = base + min(need, bseen);
  for (int i = t0; i < t1; ++i) {
    const int t = pick(i);
    if (t == 1 || (t == 2 && bseen < need)) {
      if (o < k) out[o] = s0 + i;
      ++o;
    }
    bseen += t == 2;
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
  p.rowlse = reinterpret_cast<float*>(w);
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
  // keys per scoring CTA: a whole number of 128-key tiles T, the one of least cost
  // (waves of resident CTAs, two per SM, rounded up) x (T + 2.4): a CTA's set-up is
  // worth 2.4 tiles, and a partial last wave costs as much as a full one.  The model
  // ranks 16, 23/24, 27, 32 and 35 tiles as GB300 timings did at 32K-109K prompts and
  // batches 1-16 (from 4 tiles up, within the split table).
  {
    const long slots = 2L * num_sms();
    double best_cost = -1.0;
    int best_t = 16;
    const int t_min = (Lmax_seen + kMaxSnapSplit * kTcTile - 1) / (kMaxSnapSplit * kTcTile);
    for (int t = t_min > 4 ? t_min : 4; t <= 512; ++t) {
      long items = 0;
      for (int b = 0; b < a.B; ++b) {
        const int tiles = (a.prompt_len[b] + kTcTile - 1) / kTcTile;
        items += (long)a.Hkv * ((tiles + t - 1) / t);
      }
      const double cost = (double)((items + slots - 1) / slots) * (t + 2.4);
      if (best_cost < 0.0 || cost < best_cost) {
        best_cost = cost;
        best_t = t;
      }
      if (items <= slots) break;  // one wave: larger CTAs only lengthen it
    }
    p.item_keys = best_t * kTcTile;
    // The flat split: N <= slots CTAs of equal shares of all the units' tiles (at
    // least 4 each), one wave; a share that runs into the next unit reloads the query
    // tile, worth ~1.5 tiles.  Taken when the model ranks it first: when the units'
    // tiles do not divide into the slots (64 units of 512 tiles fill 256 of 304).
    long T1 = 0;
    for (int b = 0; b < a.B; ++b) T1 += (long)a.Hkv * ((a.prompt_len[b] + kTcTile - 1) / kTcTile);
    int N = (int)(T1 / 4 < slots ? T1 / 4 : slots);
    // every unit's pass-1 statistics must fit its kMaxSnapSplit slots
    auto parts_fit = [&](int n) {
      long first = 0;
      for (int b = 0; b < a.B; ++b) {
        const long ut = (a.prompt_len[b] + kTcTile - 1) / kTcTile;
        for (int g = 0; g < a.Hkv; ++g, first += ut) {
          const long c0 = ((first + 1) * n - 1) / T1, c1 = ((first + ut) * n - 1) / T1;
          if (c1 - c0 + 1 > kMaxSnapSplit) return false;
        }
      }
      return true;
    };
    while (N > 1 && !parts_fit(N)) --N;
    p.flat = 0;
    p.flat_ctas = 0;
    if (N >= 1 && (double)T1 / N + 2.4 + 1.5 < best_cost) {
      p.flat = 1;
      p.flat_ctas = N;
    }
  }
  p.nsplit = p.flat ? kMaxSnapSplit : (Lmax_seen + p.item_keys - 1) / p.item_keys;
  if (p.nsplit > kMaxSnapSplit) {
    set_last_error("prompt longer than the scoring kernels' split table (524288 tokens)");
    return cudaErrorInvalidValue;
  }
  if (!encode_rows_map(&p.tmk, a.k, (uint64_t)a.B * a.Hkv * a.Lmax, kTcTile)) {
    set_last_error("cuTensorMapEncodeTiled failed for the prompt keys");
    return cudaErrorInvalidValue;
  }
  if (!encode_rows_map(&p.tmq, a.q_win, (uint64_t)a.B * a.Hq * a.w, kTcTile)) {
    set_last_error("cuTensorMapEncodeTiled failed for the window queries");
    return cudaErrorInvalidValue;
  }
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(snap_score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    cudaFuncSetAttribute(snap_score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    attrs = true;
  }
  // nothing to evict anywhere (RocketKV-MT's split): the kept set is every position,
  // so the scoring passes are skipped and the select only writes the identity
  bool evicts = false;
  for (int b = 0; b < a.B; ++b) evicts |= a.keep1[b] < a.prompt_len[b];
  // pass 2 scores the L - w prefix keys: in the flat split, at most one CTA a tile
  long T2 = 0;
  for (int b = 0; b < a.B; ++b)
    T2 += (long)a.Hkv * (a.prompt_len[b] > a.w ? (a.prompt_len[b] - a.w + kTcTile - 1) / kTcTile : 0);
  const dim3 sgrid = p.flat ? dim3((unsigned)p.flat_ctas) : dim3(p.nsplit, (unsigned)units);
  const dim3 sgrid2 = p.flat ? dim3((unsigned)(T2 < p.flat_ctas ? T2 : p.flat_ctas)) : sgrid;
  if (evicts) {
    launch_begin(K_SNAP_STATS, s);
    snap_score_kernel<true><<<sgrid, kTcThreads, kTcSmem, s>>>(p);
    launch_end(K_SNAP_STATS, s);
    launch_begin(K_SNAP_STATS_COMBINE, s);
    snap_stats_combine_kernel<<<(unsigned)units, 128, 0, s>>>(p);
    launch_end(K_SNAP_STATS_COMBINE, s);
    launch_begin(K_SNAP_COLSUM, s);
    if (sgrid2.x > 0) snap_score_kernel<false><<<sgrid2, kTcThreads, kTcSmem, s>>>(p);
    launch_end(K_SNAP_COLSUM, s);
    launch_begin(K_SNAP_POOL, s);
    snap_pool_kernel<<<dim3((Lmax_seen + kPoolTile - 1) / kPoolTile, (unsigned)units), kPoolThreads, 0, s>>>(p);
    launch_end(K_SNAP_POOL, s);
  }
  // select: clusters of up to 8 CTAs per unit (about 4096 prefix positions per CTA)
  // while the units alone leave SMs idle; 2 once they cover the SMs (measured: wider
  // clusters then only add cluster barriers)
  int Lp_max = 1;
  for (int b = 0; b < a.B; ++b) Lp_max = a.prompt_len[b] - a.w > Lp_max ? a.prompt_len[b] - a.w : Lp_max;
  int csel = (Lp_max + 4095) / 4096;
  int by_units = (int)((long)num_sms() / (long)units);
  by_units = by_units > 2 ? by_units : 2;
  const int by_smem = (Lp_max + kSelectSliceMax - 1) / kSelectSliceMax;  // the slices must fit
  csel = csel < by_units ? csel : by_units;
  csel = csel > by_smem ? csel : by_smem;
  csel = csel < 1 ? 1 : (csel > kSelectMaxCluster ? kSelectMaxCluster : csel);
  const int slice = (Lp_max + csel - 1) / csel;
  if (slice > kSelectSliceMax) {
    set_last_error("prompt longer than the select's shared-memory staging (393216 tokens)");
    return cudaErrorInvalidValue;
  }
  static bool sel_attr = false;
  if (!sel_attr) {
    cudaFuncSetAttribute(snap_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelectSliceMax * 4);
    sel_attr = true;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csel, (unsigned)units, 1);
    cfg.blockDim = dim3(kSelectThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)slice * 4;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csel;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    launch_begin(K_SNAP_SELECT, s);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, snap_select_kernel, p);
    launch_end(K_SNAP_SELECT, s);
    if (e != cudaSuccess) return e;
  }
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

// --------------------------------------------------------------------------
// Chunked prefill: the held survivors (read through the page table) and the new
// chunk, back to back into contiguous [B][Hkv][Lc][128] K and V in the workspace, so
// the stage-1 pipeline above can run over them.  grid (ceil(Lc / 16), Hkv, B), 256
// threads: 16 rows x 16 pieces of 16 bytes per pass.
struct GatherParams {
  const rkv_bf16* k_pages;
  const rkv_bf16* v_pages;
  const int32_t* page_table;
  const int32_t* seq_len;
  int32_t* err;
  const rkv_bf16* k_chunk;
  const rkv_bf16* v_chunk;
  rkv_bf16* k_out;
  rkv_bf16* v_out;
  int Hkv, P, max_pages, num_phys, chunk_max, Lc;
  int32_t held[RKV_MAX_BATCH];
  int32_t chunk[RKV_MAX_BATCH];
};

__global__ void __launch_bounds__(256) chunk_gather_kernel(const __grid_constant__ GatherParams p) {
  const int b = blockIdx.z, g = blockIdx.y;
  const int held = p.held[b], n = held + p.chunk[b];
  if (blockIdx.x == 0 && g == 0 && threadIdx.x == 0 && p.seq_len[b] != held) flag_error(p.err, RKV_DEVERR_SEQ_LEN);
  const int t = blockIdx.x * 16 + (threadIdx.x >> 4), piece = threadIdx.x & 15;
  if (t >= n) return;
  const rkv_bf16 *ks, *vs;
  if (t < held) {
    const int phys = p.page_table[(size_t)b * p.max_pages + t / p.P];
    if (phys < 0 || phys >= p.num_phys) {
      if (piece == 0) flag_error(p.err, RKV_DEVERR_PAGE_ID);
      return;
    }
    const size_t row = (((size_t)phys * p.Hkv + g) * p.P + t % p.P) * 128;
    ks = p.k_pages + row;
    vs = p.v_pages + row;
  } else {
    const size_t row = (((size_t)b * p.Hkv + g) * p.chunk_max + (t - held)) * 128;
    ks = p.k_chunk + row;
    vs = p.v_chunk + row;
  }
  const size_t dst = (((size_t)b * p.Hkv + g) * p.Lc + t) * 128 + piece * 8;
  *reinterpret_cast<uint4*>(p.k_out + dst) = reinterpret_cast<const uint4*>(ks)[piece];
  *reinterpret_cast<uint4*>(p.v_out + dst) = reinterpret_cast<const uint4*>(vs)[piece];
}

size_t prefill_chunk_ws_bytes(int B, int Hq, int Hkv, int w, int Lc) {
  return 2 * align256((size_t)B * Hkv * Lc * 128 * 2) + prefill_ws_bytes(B, Hq, Hkv, w, Lc);
}

cudaError_t launch_prefill_chunk(const PrefillChunkArgs& a, cudaStream_t s) {
  const rkv_cache& c = a.cache;
  int Lc = 1;
  int32_t n[RKV_MAX_BATCH], keep[RKV_MAX_BATCH];
  for (int b = 0; b < c.B; ++b) {
    n[b] = a.held_len[b] + a.chunk_len[b];
    keep[b] = a.keep1[b] < n[b] ? a.keep1[b] : n[b];
    Lc = n[b] > Lc ? n[b] : Lc;
  }
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  const size_t kv_bytes = align256((size_t)c.B * c.Hkv * Lc * 128 * 2);
  GatherParams gp;
  gp.k_pages = c.k_pages;
  gp.v_pages = c.v_pages;
  gp.page_table = c.page_table;
  gp.seq_len = c.seq_len;
  gp.err = c.error_word;
  gp.k_chunk = a.k_chunk;
  gp.v_chunk = a.v_chunk;
  gp.k_out = reinterpret_cast<rkv_bf16*>(w);
  gp.v_out = reinterpret_cast<rkv_bf16*>(w + kv_bytes);
  gp.Hkv = c.Hkv;
  gp.P = c.page_size;
  gp.max_pages = c.max_pages;
  gp.num_phys = c.num_phys_pages;
  gp.chunk_max = a.chunk_max;
  gp.Lc = Lc;
  for (int b = 0; b < c.B; ++b) {
    gp.held[b] = a.held_len[b];
    gp.chunk[b] = a.chunk_len[b];
  }
  launch_begin(K_CHUNK_GATHER, s);
  chunk_gather_kernel<<<dim3((Lc + 15) / 16, c.Hkv, c.B), 256, 0, s>>>(gp);
  launch_end(K_CHUNK_GATHER, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  PrefillArgs pa;
  pa.q_win = a.q_win;
  pa.k = gp.k_out;
  pa.v = gp.v_out;
  pa.B = c.B;
  pa.Hq = a.Hq;
  pa.Hkv = c.Hkv;
  pa.G = a.Hq / c.Hkv;
  pa.w = a.w;
  pa.Lmax = Lc;
  pa.prompt_len = n;
  pa.keep1 = keep;
  pa.pool_kernel = a.pool_kernel;
  pa.scale = a.scale;
  pa.cache = c;
  pa.kept_idx = a.kept_idx;
  pa.kept_stride = a.kept_stride;
  pa.pooled_out = nullptr;
  pa.ws = w + 2 * kv_bytes;
  pa.ws_bytes = a.ws_bytes - 2 * kv_bytes;
  return launch_prefill(pa, s);
}

}  // namespace rkv
