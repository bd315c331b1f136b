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
// The logits are m16n8k16 bf16 tensor-core MMAs with fp32 accumulation; K tiles are
// staged in shared memory with cp.async, Q fragments stay in registers.
#include "rkv_device.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

constexpr int kSnapThreads = 128;  // 4 warps x 32 query rows
constexpr int kSnapTile = 64;      // keys per shared-memory tile
constexpr int kRowB = 272;         // 256 B key row + 16 B pad
constexpr int kSnapSmem = 128 * kRowB + 2 * kSnapTile * kRowB + 4 * kSnapTile * 4;
constexpr int kMaxSnapSplit = 256;
constexpr int kPoolTile = 2048;
constexpr int kPoolThreads = 256;
constexpr int kMaxPool = 255;
constexpr int kSelectThreads = 1024;

struct SnapParams {
  const rkv_bf16* q_win;
  const rkv_bf16* k;
  const rkv_bf16* v;
  int B, Hq, Hkv, G, w, R, Lmax, nsplit, tiles_per_split;
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

// ---------------------------------------------------------------------------
// Both passes.  grid (nsplit, B*Hkv), 128 threads, dynamic smem kSnapSmem.
// Warp w owns query rows [32w, 32w+32) as two m16 tiles; a 64-key tile is 8 n8
// tiles; the 128 channels are 8 k16 steps.
// ---------------------------------------------------------------------------
template <bool kStats>
__global__ void __launch_bounds__(kSnapThreads) snap_score_kernel(const __grid_constant__ SnapParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* qs = smem;
  uint8_t* ks = smem + 128 * kRowB;
  float* colbuf = reinterpret_cast<float*>(ks + 2 * kSnapTile * kRowB);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv, split = blockIdx.x;
  const int L = p.L[b];
  const int col_end = kStats ? L : L - p.w;  // keys scored by this pass
  const int t_begin = split * p.tiles_per_split * kSnapTile;
  const int t_end = min(col_end, t_begin + p.tiles_per_split * kSnapTile);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kSnapTile - 1) / kSnapTile : 0;

  // rows of this thread: idx = mt*2 + h -> r = 32*warp + 16*mt + lane/4 + 8*h
  int rows[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) rows[i] = 32 * warp + 16 * (i >> 1) + (lane >> 2) + 8 * (i & 1);

  if (ntiles == 0) {
    if (kStats && (lane & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        p.part[((size_t)unit * p.nsplit + split) * 128 + rows[i]] = make_float2(-1e30f, 0.f);
    }
    return;
  }

  const rkv_bf16* kbase = p.k + ((size_t)b * p.Hkv + g) * p.Lmax * 128;
  auto load_tile = [&](int ti, int buf) {
    const int t0 = t_begin + ti * kSnapTile;
    for (int e = tid; e < kSnapTile * 16; e += kSnapThreads) {
      const int row = e >> 4, c16 = e & 15;
      const int t = t0 + row;
      const bool ok = t < t_end;
      cp_async16(ks + (buf * kSnapTile + row) * kRowB + c16 * 16, ok ? kbase + (size_t)t * 128 + c16 * 8 : p.k,
                 ok ? 16u : 0u);
    }
  };
  // Q rows (zero beyond R)
  for (int e = tid; e < 128 * 16; e += kSnapThreads) {
    const int r = e >> 4, c16 = e & 15;
    const bool ok = r < p.R;
    const rkv_bf16* src =
        ok ? p.q_win + (((size_t)b * p.Hq + (size_t)g * p.G + r / p.w) * p.w + r % p.w) * 128 + c16 * 8 : p.q_win;
    cp_async16(qs + r * kRowB + c16 * 16, src, ok ? 16u : 0u);
  }
  load_tile(0, 0);
  cp_async_commit();
  if (ntiles > 1) load_tile(1, 1);
  cp_async_commit();

  // per-row state
  float st_a[4], st_b[4];   // stats: (m, l); colsum: (M, 1/l)
  int lim[4];               // stats: last visible key position of the row
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = rows[i];
    if (kStats) {
      st_a[i] = -1e30f;
      st_b[i] = 0.f;
      lim[i] = r < p.R ? L - p.w + (r % p.w) : -1;
    } else {
      const float2 rs = p.rowstat[(size_t)unit * 128 + r];
      st_a[i] = rs.x;
      st_b[i] = rs.y;
      lim[i] = 0;
    }
  }

  uint32_t af[2][8][4];
  const float sl = p.scale_log2;
  for (int ti = 0; ti < ntiles; ++ti) {
    const int buf = ti & 1;
    cp_async_wait<1>();
    __syncthreads();
    if (ti == 0) {
      const uint32_t q32 = smem_u32(qs);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ldsm_x4(af[mt][kk][0], af[mt][kk][1], af[mt][kk][2], af[mt][kk][3],
                  q32 + (warp * 32 + mt * 16 + (lane & 15)) * kRowB + (kk * 16 + (lane >> 4) * 8) * 2);
    }
    float acc[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
    const uint32_t k32 = smem_u32(ks + buf * kSnapTile * kRowB);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int kk2 = 0; kk2 < 4; ++kk2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, k32 + (nt * 8 + (lane & 7)) * kRowB + (kk2 * 32 + (lane >> 3) * 8) * 2);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t* a0 = af[mt][2 * kk2];
          const uint32_t* a1 = af[mt][2 * kk2 + 1];
          mma_16816(acc[mt][nt], a0[0], a0[1], a0[2], a0[3], b0, b1);
          mma_16816(acc[mt][nt], a1[0], a1[1], a1[2], a1[3], b2, b3);
        }
      }
    }
    __syncthreads();  // every warp is done with this buffer
    if (ti + 2 < ntiles) load_tile(ti + 2, buf);
    cp_async_commit();

    const int t0 = t_begin + ti * kSnapTile + 2 * (lane & 3);
    if (kStats) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mt = i >> 1, h = i & 1;
        float z[16];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int t = t0 + nt * 8 + c;
            const float v = (t <= lim[i] && t < t_end) ? acc[mt][nt][2 * h + c] * sl : -INFINITY;
            z[nt * 2 + c] = v;
            mx = fmaxf(mx, v);
          }
        const float m_new = fmaxf(st_a[i], mx);
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) sum += exp2f(z[e] - m_new);
        st_b[i] = st_b[i] * exp2f(st_a[i] - m_new) + sum;
        st_a[i] = m_new;
      }
    } else {
      float cs[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) cs[nt][0] = cs[nt][1] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mt = i >> 1, h = i & 1;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) cs[nt][c] += exp2f(acc[mt][nt][2 * h + c] * sl - st_a[i]) * st_b[i];
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float x = cs[nt][c];
          x += __shfl_xor_sync(0xffffffffu, x, 4);
          x += __shfl_xor_sync(0xffffffffu, x, 8);
          x += __shfl_xor_sync(0xffffffffu, x, 16);
          if (lane < 4) colbuf[warp * kSnapTile + nt * 8 + 2 * lane + c] = x;
        }
      __syncthreads();
      if (tid < kSnapTile) {
        const int t = t_begin + ti * kSnapTile + tid;
        if (t < t_end)
          p.S[(size_t)unit * p.Lmax + t] =
              (colbuf[tid] + colbuf[kSnapTile + tid]) + (colbuf[2 * kSnapTile + tid] + colbuf[3 * kSnapTile + tid]);
      }
    }
  }

  if (kStats) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, st_a[i], o);
        const float lo = __shfl_xor_sync(0xffffffffu, st_b[i], o);
        const float M = fmaxf(st_a[i], mo);
        st_b[i] = st_b[i] * exp2f(st_a[i] - M) + lo * exp2f(mo - M);
        st_a[i] = M;
      }
      if ((lane & 3) == 0) p.part[((size_t)unit * p.nsplit + split) * 128 + rows[i]] = make_float2(st_a[i], st_b[i]);
    }
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

// Top keep1-w pooled prefix positions + the window.  grid B*Hkv, 1024 threads.
__global__ void __launch_bounds__(kSelectThreads) snap_select_kernel(const __grid_constant__ SnapParams p) {
  __shared__ uint32_t hist[258];
  __shared__ int scan_scratch[kSelectThreads / 32 + 1];
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
  uint32_t T;
  int need;
  block_radix_threshold<kSelectThreads>(Lp, k, [&](int i) { return float_key(pooled[i]); }, hist, &T, &need);

  const int seg = (Lp + kSelectThreads - 1) / kSelectThreads;
  const int s0 = min(Lp, tid * seg), s1 = min(Lp, s0 + seg);
  int ceq = 0;
  for (int i = s0; i < s1; ++i) ceq += float_key(pooled[i]) == T;
  int total;
  const int eq_base = block_exclusive_scan<kSelectThreads>(ceq, scan_scratch, &total);
  int csel = 0;
  for (int i = s0, er = eq_base; i < s1; ++i) {
    const uint32_t u = float_key(pooled[i]);
    if (u > T) ++csel;
    else if (u == T) { csel += er < need; ++er; }
  }
  const int out_base = block_exclusive_scan<kSelectThreads>(csel, scan_scratch, &total);
  for (int i = s0, er = eq_base, o = out_base; i < s1; ++i) {
    const uint32_t u = float_key(pooled[i]);
    bool take = u > T;
    if (u == T) { take = er < need; ++er; }
    if (take && o < k) out[o++] = i;
  }
}

// Survivors' K/V into the cache pages and their summaries.
// grid (ceil(max keep1 / P), Hkv, B), 128 threads: channel pair = tid % 64, the two
// halves of the block take alternate tokens of the page.
__global__ void __launch_bounds__(128) snap_compact_kernel(const __grid_constant__ SnapParams p) {
  __shared__ float red[4][64];
  const int b = blockIdx.z, g = blockIdx.y, pg = blockIdx.x, tid = threadIdx.x;
  const int unit = b * p.Hkv + g;
  const int n = p.keep1[b];
  if (pg == 0 && g == 0 && tid == 0) p.seq_len[b] = n;
  if (pg * p.P >= n) return;
  const int phys = p.page_table[(size_t)b * p.max_pages + pg];
  if (phys < 0 || phys >= p.num_phys) {
    if (tid == 0) flag_error(p.err, RKV_DEVERR_PAGE_ID);
    return;
  }
  const int c2 = tid & 63, half = tid >> 6;
  const int32_t* kept = p.kept + (size_t)unit * p.kept_stride;
  const size_t src_base = ((size_t)b * p.Hkv + g) * p.Lmax * 128 + 2 * c2;
  const size_t dst_base = (((size_t)phys * p.Hkv + g) * p.P) * 128 + 2 * c2;
  float mx0 = -INFINITY, mx1 = -INFINITY, mn0 = INFINITY, mn1 = INFINITY;
  const int end = min(n, (pg + 1) * p.P);
  const int L = p.L[b];
  for (int i = pg * p.P + half; i < end; i += 2) {
    const int t = kept[i];
    if (t < 0 || t >= L) {   // never expected: the select kernel writes every position
      flag_error(p.err, RKV_DEVERR_CAPACITY);
      continue;
    }
    const size_t src = src_base + (size_t)t * 128;
    const uint32_t ku = *reinterpret_cast<const uint32_t*>(p.k + src);
    const uint32_t vu = *reinterpret_cast<const uint32_t*>(p.v + src);
    const size_t dst = dst_base + (size_t)(i - pg * p.P) * 128;
    *reinterpret_cast<uint32_t*>(p.k_pages + dst) = ku;
    *reinterpret_cast<uint32_t*>(p.v_pages + dst) = vu;
    const float x0 = bf16_lo(ku), x1 = bf16_hi(ku);
    mx0 = fmaxf(mx0, x0);
    mx1 = fmaxf(mx1, x1);
    mn0 = fminf(mn0, x0);
    mn1 = fminf(mn1, x1);
  }
  if (half == 1) {
    red[0][c2] = mx0;
    red[1][c2] = mx1;
    red[2][c2] = mn0;
    red[3][c2] = mn1;
  }
  __syncthreads();
  if (half == 0) {
    mx0 = fmaxf(mx0, red[0][c2]);
    mx1 = fmaxf(mx1, red[1][c2]);
    mn0 = fminf(mn0, red[2][c2]);
    mn1 = fminf(mn1, red[3][c2]);
    const size_t row = ((size_t)unit * 128 + 2 * c2) * p.max_pages + pg;
    p.kmax[row] = (rkv_bf16)(__float_as_uint(mx0) >> 16);
    p.kmax[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mx1) >> 16);
    p.kmin[row] = (rkv_bf16)(__float_as_uint(mn0) >> 16);
    p.kmin[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mn1) >> 16);
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
  // splits along L: one wave of 2 resident CTAs per SM (the register count allows 2)
  const int tiles = (Lmax_seen + kSnapTile - 1) / kSnapTile;
  const int slots = 2 * num_sms();
  int nsplit = (int)units < slots ? slots / (int)units : 1;
  nsplit = nsplit < 1 ? 1 : (nsplit > kMaxSnapSplit ? kMaxSnapSplit : nsplit);
  nsplit = nsplit > tiles ? tiles : nsplit;
  p.tiles_per_split = (tiles + nsplit - 1) / nsplit;
  p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;

  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(snap_score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSnapSmem);
    cudaFuncSetAttribute(snap_score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSnapSmem);
    attrs = true;
  }
  const dim3 sgrid(p.nsplit, (unsigned)units);
  launch_begin(K_SNAP_STATS, s);
  snap_score_kernel<true><<<sgrid, kSnapThreads, kSnapSmem, s>>>(p);
  launch_end(K_SNAP_STATS, s);
  launch_begin(K_SNAP_STATS_COMBINE, s);
  snap_stats_combine_kernel<<<(unsigned)units, 128, 0, s>>>(p);
  launch_end(K_SNAP_STATS_COMBINE, s);
  launch_begin(K_SNAP_COLSUM, s);
  snap_score_kernel<false><<<sgrid, kSnapThreads, kSnapSmem, s>>>(p);
  launch_end(K_SNAP_COLSUM, s);
  launch_begin(K_SNAP_POOL, s);
  snap_pool_kernel<<<dim3((Lmax_seen + kPoolTile - 1) / kPoolTile, (unsigned)units), kPoolThreads, 0, s>>>(p);
  launch_end(K_SNAP_POOL, s);
  launch_begin(K_SNAP_SELECT, s);
  snap_select_kernel<<<(unsigned)units, kSelectThreads, 0, s>>>(p);
  launch_end(K_SNAP_SELECT, s);
  launch_begin(K_SNAP_COMPACT, s);
  snap_compact_kernel<<<dim3((keep_max + p.P - 1) / p.P, a.Hkv, a.B), 128, 0, s>>>(p);
  launch_end(K_SNAP_COMPACT, s);
  return cudaGetLastError();
}

}  // namespace rkv
