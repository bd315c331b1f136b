// Exact-TopK recall of a decode step's page selection (a diagnostic, not on the hot
// path).
//
// The summary page of "RocketKV: Accelerating Long-Context LLM Inference via
// Two-Stage KV Cache Compression" measures RocketKV against the Exact-TopK baseline
// ("Surprising findings", "Limitations"); "RocketKV-adapted" (VeloxQuant-MLX docs)
// compares selections with an oracle top-k ("Where it sits -- the mechanism gap")
// and by selection overlap ("Evidence").  For one (sequence, KV head) this kernel
// scores every cached token exactly, e_t = sum over the group's heads of
// softmax_t(q_h . k_t * scale), takes the K largest (ties: lower index), and counts
// how many of them, and how much of their mass, lie in the selected pages.
//
// One CTA per (sequence, KV head), 512 threads (a warp per token at a time): pass 1
// reads each token's key row through the page table and keeps per-head running max /
// sum; pass 2 recomputes the logits and stages e_t as order-preserving keys in shared
// memory; the block select of the decode path picks the top K and the counts ride on
// its output callback.
#include "rkv_device.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

constexpr int kDiagThreads = 512;
constexpr int kDiagMaxTokens = 48 * 1024;  // keys staged in shared memory (192 KB)

struct RecallParams {
  const rkv_bf16* k_pages;
  const int32_t* page_table;
  const int32_t* seq_len;
  const rkv_bf16* q;
  const int32_t* sel_pages;
  int sel_stride;
  float* recall;
  float* mass;
  int32_t* err;
  int B, Hkv, Hq, G, P, max_pages, num_phys;
  float scale_log2;
  int32_t k_tokens[RKV_MAX_BATCH];
};

// Logits of token t for the group's G heads, scaled to base 2, in every lane of the
// calling warp; false if the token's page id is invalid.  Lane l holds channels
// 4l .. 4l+3 of each head's query (qr) and reads the same channels of the key row, so
// the warp reads the row as one coalesced 256-byte line; a butterfly sums the lanes.
template <int G>
__device__ __forceinline__ bool token_logits(const RecallParams& p, int b, int g, int t, const float (&qr)[G][4],
                                             float (&z)[G]) {
  const int lane = threadIdx.x & 31;
  const int phys = p.page_table[(size_t)b * p.max_pages + t / p.P];
  if (phys < 0 || phys >= p.num_phys) return false;
  const uint2 kv =
      reinterpret_cast<const uint2*>(p.k_pages + (((size_t)phys * p.Hkv + g) * p.P + t % p.P) * 128)[lane];
  const float k0 = bf16_lo(kv.x), k1 = bf16_hi(kv.x), k2 = bf16_lo(kv.y), k3 = bf16_hi(kv.y);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = qr[h][0] * k0;
    x = fmaf(qr[h][1], k1, x);
    x = fmaf(qr[h][2], k2, x);
    x = fmaf(qr[h][3], k3, x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    z[h] = x * p.scale_log2;
  }
  return true;
}

// One CTA per (sequence, KV head); warp w scores tokens w, w + 16, ...
template <int G>
__global__ void __launch_bounds__(kDiagThreads) recall_kernel(const __grid_constant__ RecallParams p) {
  extern __shared__ uint32_t sk[];  // [n] keys of e_t
  __shared__ float wm[8][kDiagThreads / 32], wl[8][kDiagThreads / 32];
  __shared__ float hM[8], hinvL[8];
  __shared__ uint32_t pagebit[kDiagMaxTokens / 16 / 32];
  __shared__ TopkSmem<kDiagThreads> ts;
  __shared__ float red[3][kDiagThreads / 32];
  constexpr int NW = kDiagThreads / 32;
  const int unit = blockIdx.x, b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int n = p.seq_len[b];
  const int cap = min(p.max_pages * p.P, kDiagMaxTokens);
  if (n < 0 || n > cap) {
    if (tid == 0) flag_error(p.err, RKV_DEVERR_CAPACITY);
    n = n < 0 ? 0 : cap;
  }
  const int K = min(p.k_tokens[b], n);
  float qr[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint2 qv = reinterpret_cast<const uint2*>(p.q + ((size_t)b * p.Hq + (size_t)g * G + h) * 128)[lane];
    qr[h][0] = bf16_lo(qv.x);
    qr[h][1] = bf16_hi(qv.x);
    qr[h][2] = bf16_lo(qv.y);
    qr[h][3] = bf16_hi(qv.y);
  }
  const int NP = (n + p.P - 1) / p.P;
  for (int i = tid; i < (NP + 31) / 32; i += kDiagThreads) pagebit[i] = 0u;
  __syncthreads();
  // the selected pages (ascending, ended by -1 or the row's end)
  for (int i = tid; i < p.sel_stride; i += kDiagThreads) {
    const int pg = p.sel_pages[(size_t)unit * p.sel_stride + i];
    if (pg >= 0 && pg < NP) atomicOr(&pagebit[pg >> 5], 1u << (pg & 31));
  }
  // pass 1: per-head max and sum of 2^z over the tokens (identical in every lane)
  float m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  bool bad = false;
  for (int t = warp; t < n; t += NW) {
    float z[G];
    if (!token_logits<G>(p, b, g, t, qr, z)) {
      bad = true;
      continue;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mn = fmaxf(m[h], z[h]);
      l[h] = l[h] * exp2f(m[h] - mn) + exp2f(z[h] - mn);
      m[h] = mn;
    }
  }
  if (bad && lane == 0) flag_error(p.err, RKV_DEVERR_PAGE_ID);
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      wm[h][warp] = m[h];
      wl[h][warp] = l[h];
    }
  }
  __syncthreads();
  if (tid < G) {
    float mm = -INFINITY, ll = 0.f;
    for (int w = 0; w < NW; ++w) mm = fmaxf(mm, wm[tid][w]);
    for (int w = 0; w < NW; ++w)
      if (wm[tid][w] != -INFINITY) ll += wl[tid][w] * exp2f(wm[tid][w] - mm);
    hM[tid] = mm;
    hinvL[tid] = ll > 0.f ? 1.f / ll : 0.f;
  }
  __syncthreads();
  // pass 2: e_t as keys (e_t >= 0, so its key is its bit pattern with the top bit set)
  for (int t = warp; t < n; t += NW) {
    float z[G];
    float e = 0.f;
    if (token_logits<G>(p, b, g, t, qr, z)) {
#pragma unroll
      for (int h = 0; h < G; ++h) e += exp2f(z[h] - hM[h]) * hinvL[h];
    }
    if (lane == 0) sk[t] = float_key(e);
  }
  __syncthreads();
  // top K and the counts
  float hit = 0.f, mh = 0.f, mt = 0.f;
  auto count = [&](int i) {
    const float e = __uint_as_float(sk[i] & 0x7fffffffu);
    const bool in = (pagebit[(i / p.P) >> 5] >> ((i / p.P) & 31)) & 1u;
    hit += in ? 1.f : 0.f;
    mh += in ? e : 0.f;
    mt += e;
  };
  if (K >= n) {
    for (int i = tid; i < n; i += kDiagThreads) count(i);
  } else if (K > 0) {
    topk_adaptive_fn<kDiagThreads>(n, K, [&](int i) { return sk[i]; }, ts, [&](int, int i) { count(i); });
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    hit += __shfl_xor_sync(0xffffffffu, hit, o);
    mh += __shfl_xor_sync(0xffffffffu, mh, o);
    mt += __shfl_xor_sync(0xffffffffu, mt, o);
  }
  if (lane == 0) {
    red[0][warp] = hit;
    red[1][warp] = mh;
    red[2][warp] = mt;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, bm = 0.f, c = 0.f;
    for (int w = 0; w < NW; ++w) {
      a += red[0][w];
      bm += red[1][w];
      c += red[2][w];
    }
    p.recall[unit] = K > 0 ? a / (float)K : 1.f;
    if (p.mass) p.mass[unit] = c > 0.f ? bm / c : 1.f;
  }
}

}  // namespace

int recall_max_tokens() { return kDiagMaxTokens; }

cudaError_t launch_recall(const RecallArgs& a, cudaStream_t s) {
  RecallParams p;
  p.k_pages = a.cache.k_pages;
  p.page_table = a.cache.page_table;
  p.seq_len = a.cache.seq_len;
  p.q = a.q;
  p.sel_pages = a.sel_pages;
  p.sel_stride = a.sel_pages_stride;
  p.recall = a.recall;
  p.mass = a.mass;
  p.err = a.cache.error_word;
  p.B = a.cache.B;
  p.Hkv = a.cache.Hkv;
  p.Hq = a.Hq;
  p.G = a.Hq / a.cache.Hkv;
  p.P = a.cache.page_size;
  p.max_pages = a.cache.max_pages;
  p.num_phys = a.cache.num_phys_pages;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  for (int b = 0; b < a.cache.B; ++b) p.k_tokens[b] = a.k_tokens[b];
  const int cap = a.cache.max_pages * a.cache.page_size;
  const size_t smem = (size_t)(cap < kDiagMaxTokens ? cap : kDiagMaxTokens) * 4;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(recall_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDiagMaxTokens * 4);
    cudaFuncSetAttribute(recall_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDiagMaxTokens * 4);
    cudaFuncSetAttribute(recall_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDiagMaxTokens * 4);
    cudaFuncSetAttribute(recall_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDiagMaxTokens * 4);
    attr = true;
  }
  const unsigned grid = a.cache.B * a.cache.Hkv;
  launch_begin(K_RECALL, s);
  if (p.G == 1)
    recall_kernel<1><<<grid, kDiagThreads, smem, s>>>(p);
  else if (p.G == 2)
    recall_kernel<2><<<grid, kDiagThreads, smem, s>>>(p);
  else if (p.G == 4)
    recall_kernel<4><<<grid, kDiagThreads, smem, s>>>(p);
  else
    recall_kernel<8><<<grid, kDiagThreads, smem, s>>>(p);
  launch_end(K_RECALL, s);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self-test of the failure path every kernel shares: one thread waits on an mbarrier
// that nothing arrives on and no copy completes, so the bounded wait must run out; it
// then flags RKV_DEVERR_TIMEOUT exactly as a stalled ring would.  Nothing is in
// flight on the barrier, so the CTA may exit at once.
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, limit_ns)) flag_error(err, RKV_DEVERR_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_selftest(int32_t* err, uint64_t limit_ns, cudaStream_t s) {
  launch_begin(K_WAIT_SELFTEST, s);
  wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  launch_end(K_WAIT_SELFTEST, s);
  return cudaGetLastError();
}

}  // namespace rkv
