// Stage 2 of RocketKV: one Hybrid Sparse Attention (HSA) decode step.
//
// "RocketKV-adapted -- Two-Stage Compression" (VeloxQuant-MLX docs), section
// "Where it sits -- the mechanism gap": HSA bounds each page's score from
// Quest-style paged element-wise max/min summaries along the sequence, restricted
// to the SparQ-style top-magnitude channels of the query along the head dimension;
// section "Adaptation notes": whole pages (k2 of them) are selected and attended.
//
// Four kernels per step, all on the caller's stream:
//   hsa_score   channel select (top-k1 of sum_h |q_h|) + page bound s_p for every page
//   hsa_topk    block radix select of the top-k2 pages, (s_p desc, page asc)
//   hsa_attend  split flash-decode over the selected pages: bulk (TMA engine) copies
//               of 16-token K/V chunks into shared memory, m16n8k16 bf16 tensor-core
//               MMAs for q.K^T and P.V, fp32 online softmax
//   hsa_combine merge of the splits (only when the attention is split)
#include <climits>

#include "rkv_device.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

constexpr int kMaxSplit = 64;
constexpr int kScoreThreads = 256;
constexpr int kScorePages = 2 * kScoreThreads;  // pages scored per CTA (2 per thread)
constexpr int kTopkThreads = 1024;
constexpr int kAtWarps = 4;
constexpr int kAtStages = 3;
constexpr int kChunkTok = 16;                        // tokens per pipeline stage
constexpr int kRowBytes = 272;                       // 256 B token row + 16 B pad
constexpr int kStageBytes = 2 * kChunkTok * kRowBytes;  // K rows then V rows
constexpr int kAtCombineBytes = kAtWarps * 8 * (2 + 128) * 4;
constexpr int kAttendSmem = kAtWarps * kAtStages * kStageBytes + kAtCombineBytes;

struct HsaParams {
  const rkv_bf16* k_pages;
  const rkv_bf16* v_pages;
  const int32_t* page_table;
  const int32_t* seq_len;
  const rkv_bf16* kmax;
  const rkv_bf16* kmin;
  int32_t* err;
  const rkv_bf16* q;
  float* sigma;     // [units][max_pages]
  int32_t* selp;    // [units][max_pages]
  float* part_o;    // [B*Hq][nsplit][128]
  float2* part_ml;  // [B*Hq][nsplit]
  float* out;       // [B*Hq][128]
  int32_t* sel_channels;
  int32_t* sel_pages;
  int sel_pages_stride;
  int B, Hkv, Hq, G, P, max_pages, num_phys, nsplit;
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

// ---------------------------------------------------------------------------
// Steps 1-2: channel selection and page score bound.
// grid (ceil(max_pages / 512), B*Hkv), 256 threads; each thread scores 2 pages.
// The page bound uses max(q*Kmax, q*Kmin) = q*Kmax for q >= 0 and q*Kmin otherwise,
// so sum_h max(q_h Kmax, q_h Kmin) = Kmax * sum_h max(q_h, 0) + Kmin * sum_h min(q_h, 0).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScoreThreads) hsa_score_kernel(const __grid_constant__ HsaParams p) {
  __shared__ float qf[8][128];
  __shared__ double a[128];
  __shared__ int sel_flag[128];
  __shared__ int chan[128];
  __shared__ float qpos[128], qneg[128];

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
  __syncthreads();

  const int k1 = p.k1[b];
  if (tid < 128) {
    // channel score in fp64: a sum of <= 8 bf16 magnitudes is exact
    double s = 0.0;
    for (int h = 0; h < G; ++h) s += fabs((double)qf[h][tid]);
    a[tid] = s;
  }
  __syncthreads();
  if (tid < 128) {
    const double ai = a[tid];
    int rank = 0;
    for (int j = 0; j < 128; ++j) {
      const double aj = a[j];
      rank += (aj > ai) || (aj == ai && j < tid);
    }
    sel_flag[tid] = rank < k1;
  }
  __syncthreads();
  if (tid < 128 && sel_flag[tid]) {
    int pos = 0;
    for (int j = 0; j < tid; ++j) pos += sel_flag[j];
    chan[pos] = tid;
    float sp = 0.f, sn = 0.f;
    for (int h = 0; h < G; ++h) {
      const float x = qf[h][tid];
      sp += fmaxf(x, 0.f);
      sn += fminf(x, 0.f);
    }
    qpos[pos] = sp;
    qneg[pos] = sn;
  }
  __syncthreads();
  if (write_ch && tid < 128) p.sel_channels[(size_t)unit * 128 + tid] = tid < k1 ? chan[tid] : -1;

  const int pg = page0 + 2 * tid;
  if (pg < NP) {
    const size_t base = (size_t)unit * 128 * p.max_pages + pg;
    const rkv_bf16* mxp = p.kmax + base;
    const rkv_bf16* mnp = p.kmin + base;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < k1; ++kk) {
      const size_t off = (size_t)chan[kk] * p.max_pages;
      const uint32_t hi = __ldg(reinterpret_cast<const unsigned int*>(mxp + off));
      const uint32_t lo = __ldg(reinterpret_cast<const unsigned int*>(mnp + off));
      const float qp = qpos[kk], qn = qneg[kk];
      s0 = fmaf(qp, bf16_lo(hi), s0);
      s0 = fmaf(qn, bf16_lo(lo), s0);
      s1 = fmaf(qp, bf16_hi(hi), s1);
      s1 = fmaf(qn, bf16_hi(lo), s1);
    }
    float* sg = p.sigma + (size_t)unit * p.max_pages;
    sg[pg] = s0;
    if (pg + 1 < NP) sg[pg + 1] = s1;
  }
}

// ---------------------------------------------------------------------------
// Step 3: top-k2 pages by (score desc, page asc), written ascending.
// grid B*Hkv, 1024 threads, dynamic shared memory = max_pages keys.
// ---------------------------------------------------------------------------
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

  uint32_t T;
  int need;
  block_radix_threshold<kTopkThreads>(NP, k, [&](int i) { return keys[i]; }, hist, &T, &need);

  const int seg = (NP + kTopkThreads - 1) / kTopkThreads;
  const int s0 = min(NP, tid * seg), s1 = min(NP, s0 + seg);
  int ceq = 0;
  for (int i = s0; i < s1; ++i) ceq += keys[i] == T;
  int total;
  const int eq_base = block_exclusive_scan<kTopkThreads>(ceq, scan_scratch, &total);
  int csel = 0;
  for (int i = s0, er = eq_base; i < s1; ++i) {
    const uint32_t u = keys[i];
    if (u > T) ++csel;
    else if (u == T) { csel += er < need; ++er; }
  }
  const int out_base = block_exclusive_scan<kTopkThreads>(csel, scan_scratch, &total);
  for (int i = s0, er = eq_base, o = out_base; i < s1; ++i) {
    const uint32_t u = keys[i];
    bool take = u > T;
    if (u == T) { take = er < need; ++er; }
    if (take && o < k) {
      out[o] = i;
      if (user) user[o] = i;
      ++o;
    }
  }
}

// ---------------------------------------------------------------------------
// Step 4: exact softmax attention over the selected pages, split across CTAs.
// grid (nsplit, B*Hkv), 4 warps.  The unit's selected pages are cut into 16-token
// chunks ("items"); the CTA takes a contiguous range of items and its warps take
// every 4th one.  Each warp runs its own 3-stage ring: one bulk copy per lane (16 K
// rows + 16 V rows of 256 B, into 272-B padded rows so ldmatrix is conflict free),
// completion on one mbarrier per stage.  Query heads of the GQA group are the M
// rows of the MMAs (G <= 8 of 16 used).  P is split into bf16 hi + lo parts so the
// P.V product keeps ~16 bits of the fp32 probabilities.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAtWarps * 32) hsa_attend_kernel(const __grid_constant__ HsaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kAtWarps][kAtStages];
  __shared__ int tstart[kAtWarps][kAtStages];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.y, b = unit / p.Hkv, g = unit % p.Hkv, split = blockIdx.x;
  const int P = p.P, G = p.G;
  const int n = seq_length(p, b);
  const int NP = (n + P - 1) / P;
  const int k = min(p.k2[b], NP);
  const int cpp = P / kChunkTok;
  const int items = k * cpp;
  const int ips = (items + p.nsplit - 1) / p.nsplit;
  const int it0 = min(items, split * ips), it1 = min(items, it0 + ips);
  const int mine = it1 - it0 - warp;
  const int nj = mine > 0 ? (mine + kAtWarps - 1) / kAtWarps : 0;

  uint8_t* wbuf = smem + warp * (kAtStages * kStageBytes);
  const int32_t* selp = p.selp + (size_t)unit * p.max_pages;
  const int32_t* ptab = p.page_table + (size_t)b * p.max_pages;

  // query fragments (A operand rows = heads of the group)
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
    for (int s = 0; s < kAtStages; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int j) {
    const int s = j % kAtStages;
    const int it = it0 + warp + j * kAtWarps;
    int page = selp[it / cpp];
    const int chunk = it % cpp;
    const bool page_ok = page >= 0 && page < NP;   // always true for the top-k kernel's output
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
      tstart[warp][s] = t0;
      mbar_arrive_expect_tx(&bars[warp][s], 2 * kChunkTok * 256);
    }
    __syncwarp();
    const rkv_bf16* src = lane < 16 ? p.k_pages + off + lane * 128 : p.v_pages + off + (lane - 16) * 128;
    bulk_g2s(wbuf + s * kStageBytes + lane * kRowBytes, src, 256, &bars[warp][s]);
  };

  float m_run = -1e30f, l_run = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int pre = min(nj, kAtStages);
  for (int j = 0; j < pre; ++j) issue(j);
  int issued = pre, consumed = 0;

  int timed_out = 0;
  const float sl = p.scale_log2;
  for (int j = 0; j < nj; ++j) {
    const int s = j % kAtStages;
    if (!mbar_wait(&bars[warp][s], (uint32_t)((j / kAtStages) & 1))) {
      flag_error(p.err, RKV_DEVERR_TIMEOUT);
      timed_out = 1;
      break;
    }
    uint8_t* kb = wbuf + s * kStageBytes;
    uint8_t* vb = kb + kChunkTok * kRowBytes;
    const int nvalid = n - tstart[warp][s];
    if (nvalid < kChunkTok) {
      // rows past the end of the sequence hold stale data: zero their V rows
      const int nv = max(nvalid, 0);
      for (int w16 = lane; w16 < (kChunkTok - nv) * 16; w16 += 32)
        *reinterpret_cast<uint4*>(vb + (nv + (w16 >> 4)) * kRowBytes + (w16 & 15) * 16) = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      __syncwarp();
    }
    // S = Q K^T over 16 tokens
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
    float z0 = (c0 < nvalid) ? sacc[0][0] * sl : -INFINITY;
    float z1 = (c0 + 1 < nvalid) ? sacc[0][1] * sl : -INFINITY;
    float z2 = (c0 + 8 < nvalid) ? sacc[1][0] * sl : -INFINITY;
    float z3 = (c0 + 9 < nvalid) ? sacc[1][1] * sl : -INFINITY;
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
    if (j + kAtStages < nj) {
      issue(j + kAtStages);
      issued = j + kAtStages + 1;
    }
  }

  if (__syncthreads_or(timed_out)) {
    // wait (bounded) for this warp's copies still in flight, then give up
    for (int j = consumed; j < issued; ++j) mbar_wait(&bars[warp][j % kAtStages], (uint32_t)((j / kAtStages) & 1));
    return;
  }

  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

  // combine the 4 warps: [warp][head] (m, l) and [warp][head][128] o
  float* cm = reinterpret_cast<float*>(smem + kAtWarps * kAtStages * kStageBytes);
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
  const int c = threadIdx.x;  // channel
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
    const size_t bh = (size_t)b * p.Hq + (size_t)g * G + h;
    if (p.nsplit == 1) {
      p.out[bh * 128 + c] = L > 0.f ? O / L : 0.f;
    } else {
      p.part_o[(bh * p.nsplit + split) * 128 + c] = O;
      if (c == 0) p.part_ml[bh * p.nsplit + split] = make_float2(M, L);
    }
  }
}

// Merge of the attention splits.  grid B*Hq, 128 threads (one per channel).
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

}  // namespace

size_t decode_ws_bytes(int B, int Hq, int Hkv, int max_pages) {
  const size_t units = (size_t)B * Hkv;
  return align256(units * max_pages * 4) * 2 + align256((size_t)B * Hq * kMaxSplit * 128 * 4) +
         align256((size_t)B * Hq * kMaxSplit * 8);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const rkv_cache& c = a.cache;
  HsaParams p;
  p.k_pages = c.k_pages;
  p.v_pages = c.v_pages;
  p.page_table = c.page_table;
  p.seq_len = c.seq_len;
  p.kmax = c.kmax;
  p.kmin = c.kmin;
  p.err = c.error_word;
  p.q = a.q;
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  const size_t units = (size_t)c.B * c.Hkv;
  p.sigma = reinterpret_cast<float*>(w);
  w += align256(units * c.max_pages * 4);
  p.selp = reinterpret_cast<int32_t*>(w);
  w += align256(units * c.max_pages * 4);
  p.part_o = reinterpret_cast<float*>(w);
  w += align256((size_t)c.B * a.Hq * kMaxSplit * 128 * 4);
  p.part_ml = reinterpret_cast<float2*>(w);
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
  int k2max = 1;
  for (int b = 0; b < c.B; ++b) {
    p.k1[b] = a.k1[b];
    p.k2[b] = a.k2[b];
    k2max = a.k2[b] > k2max ? a.k2[b] : k2max;
  }
  const int items = (k2max < c.max_pages ? k2max : c.max_pages) * (c.page_size / kChunkTok);
  int nsplit = (4 * num_sms() + (int)units - 1) / (int)units;
  const int by_items = (items + kAtWarps - 1) / kAtWarps;
  nsplit = nsplit < by_items ? nsplit : by_items;
  nsplit = nsplit < 1 ? 1 : (nsplit > kMaxSplit ? kMaxSplit : nsplit);
  p.nsplit = nsplit;

  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(hsa_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttendSmem);
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
  hsa_attend_kernel<<<dim3(nsplit, (unsigned)units), kAtWarps * 32, kAttendSmem, s>>>(p);
  launch_end(K_HSA_ATTEND, s);
  if (nsplit > 1) {
    launch_begin(K_HSA_COMBINE, s);
    hsa_combine_kernel<<<(unsigned)(c.B * a.Hq), 128, 0, s>>>(p);
    launch_end(K_HSA_COMBINE, s);
  }
  return cudaGetLastError();
}

}  // namespace rkv
