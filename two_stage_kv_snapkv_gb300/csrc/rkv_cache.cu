// Paged cache append and Kmax/Kmin page summaries.
//
// "RocketKV-adapted -- Two-Stage Compression" (VeloxQuant-MLX docs): section
// "Where it sits -- the mechanism gap" (Quest-style paged element-wise max/min
// summaries along the sequence) and section "Evidence" (the incremental update at
// decode equals a rebuild of the summaries, bit for bit).  Min and max of bf16
// values are exact, so folding new tokens into a page's stored summary, or
// recomputing the page from its tokens, is bit-identical to any rebuild order.
#include "rkv_device.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

struct AppendParams {
  rkv_bf16* k_pages;
  rkv_bf16* v_pages;
  const int32_t* page_table;
  int32_t* seq_len;
  rkv_bf16* kmax;
  rkv_bf16* kmin;
  int32_t* err;
  const rkv_bf16* k_new;  // [B][Hkv][n_new][128] or null
  const rkv_bf16* v_new;
  int B, Hkv, P, max_pages, num_phys, n_new;
};

// Writes the summary of page `pg` of (b, g) for the channel pair (2*c2, 2*c2+1)
// from its first `cnt` tokens.
__device__ __forceinline__ void summarize_pair(const AppendParams& p, int b, int g, int pg, int phys,
                                               int cnt, int c2) {
  const rkv_bf16* base = p.k_pages + (((size_t)phys * p.Hkv + g) * p.P) * 128 + 2 * c2;
  float mx0 = -INFINITY, mx1 = -INFINITY, mn0 = INFINITY, mn1 = INFINITY;
  for (int t = 0; t < cnt; ++t) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(base + (size_t)t * 128);
    const float x0 = bf16_lo(u), x1 = bf16_hi(u);
    mx0 = fmaxf(mx0, x0);
    mx1 = fmaxf(mx1, x1);
    mn0 = fminf(mn0, x0);
    mn1 = fminf(mn1, x1);
  }
  const size_t row = ((size_t)(b * p.Hkv + g) * 128 + 2 * c2) * p.max_pages + pg;
  // the values came from bf16 bit patterns, so the top 16 bits are exact
  p.kmax[row] = (rkv_bf16)(__float_as_uint(mx0) >> 16);
  p.kmax[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mx1) >> 16);
  p.kmin[row] = (rkv_bf16)(__float_as_uint(mn0) >> 16);
  p.kmin[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mn1) >> 16);
}

// Folds new tokens [s0, s1) of page `pg` of (b, g) into the page's summary for the
// channel pair (2*c2, 2*c2+1); the keys come from k_new (token t is its row t - n).
// A page that held tokens before s0 starts from its stored summary.
__device__ __forceinline__ void fold_new_pair(const AppendParams& p, int b, int g, int pg, int n, int s0, int s1,
                                              int c2) {
  const size_t row = ((size_t)(b * p.Hkv + g) * 128 + 2 * c2) * p.max_pages + pg;
  float mx0 = -INFINITY, mx1 = -INFINITY, mn0 = INFINITY, mn1 = INFINITY;
  if (s0 > pg * p.P) {
    mx0 = bf16_f(p.kmax[row]);
    mx1 = bf16_f(p.kmax[row + p.max_pages]);
    mn0 = bf16_f(p.kmin[row]);
    mn1 = bf16_f(p.kmin[row + p.max_pages]);
  }
  const rkv_bf16* src = p.k_new + ((size_t)(b * p.Hkv + g) * p.n_new) * 128 + 2 * c2;
  for (int t = s0; t < s1; ++t) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(src + (size_t)(t - n) * 128);
    const float x0 = bf16_lo(u), x1 = bf16_hi(u);
    mx0 = fmaxf(mx0, x0);
    mx1 = fmaxf(mx1, x1);
    mn0 = fminf(mn0, x0);
    mn1 = fminf(mn1, x1);
  }
  p.kmax[row] = (rkv_bf16)(__float_as_uint(mx0) >> 16);
  p.kmax[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mx1) >> 16);
  p.kmin[row] = (rkv_bf16)(__float_as_uint(mn0) >> 16);
  p.kmin[row + p.max_pages] = (rkv_bf16)(__float_as_uint(mn1) >> 16);
}

__device__ __forceinline__ bool phys_ok(const AppendParams& p, int phys) {
  if (phys < 0 || phys >= p.num_phys) {
    flag_error(p.err, RKV_DEVERR_PAGE_ID);
    return false;
  }
  return true;
}

// Few tokens per sequence (decode): one CTA per sequence does copy, summaries and
// the length update.  With the new keys given, the touched pages' summaries fold
// them in (no page is re-read); without (the tokens were written by the caller),
// each touched page is recomputed from its tokens.  grid B, 256 threads.
__global__ void __launch_bounds__(256) append_small_kernel(const __grid_constant__ AppendParams p) {
  __shared__ int s_n;
  const int b = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) {
    const int n = p.seq_len[b];
    const bool ok = n >= 0 && n + p.n_new <= p.max_pages * p.P;
    if (!ok) flag_error(p.err, RKV_DEVERR_CAPACITY);
    s_n = ok ? n : -1;
  }
  __syncthreads();
  const int n = s_n;
  if (n < 0) return;
  const int32_t* ptab = p.page_table + (size_t)b * p.max_pages;
  if (p.k_new) {
    const int per = p.n_new * 64;
    for (int e = tid; e < p.Hkv * per; e += 256) {
      const int g = e / per, i = (e / 64) % p.n_new, c2 = e % 64;
      const int pos = n + i;
      const int phys = ptab[pos / p.P];
      if (!phys_ok(p, phys)) continue;
      const size_t dst = (((size_t)phys * p.Hkv + g) * p.P + pos % p.P) * 128 + 2 * c2;
      const size_t src = (((size_t)b * p.Hkv + g) * p.n_new + i) * 128 + 2 * c2;
      *reinterpret_cast<uint32_t*>(p.k_pages + dst) = *reinterpret_cast<const uint32_t*>(p.k_new + src);
      *reinterpret_cast<uint32_t*>(p.v_pages + dst) = *reinterpret_cast<const uint32_t*>(p.v_new + src);
    }
  }
  const int end = n + p.n_new;
  const int first = n / p.P, last = (end - 1) / p.P;
  const int per = (last - first + 1) * 64;
  if (p.k_new) {
    for (int e = tid; e < p.Hkv * per; e += 256) {
      const int g = e / per, pg = first + (e / 64) % (last - first + 1), c2 = e % 64;
      if (!phys_ok(p, ptab[pg])) continue;
      fold_new_pair(p, b, g, pg, n, max(n, pg * p.P), min(end, (pg + 1) * p.P), c2);
    }
  } else {
    __syncthreads();
    for (int e = tid; e < p.Hkv * per; e += 256) {
      const int g = e / per, pg = first + (e / 64) % (last - first + 1), c2 = e % 64;
      const int phys = ptab[pg];
      if (!phys_ok(p, phys)) continue;
      const int cnt = min(p.P, end - pg * p.P);
      summarize_pair(p, b, g, pg, phys, cnt, c2);
    }
  }
  __syncthreads();
  if (tid == 0) p.seq_len[b] = end;
}

// Many tokens: one CTA per touched (page, KV head, sequence).  grid (pages, Hkv, B),
// 128 threads; the length update runs afterwards in append_advance_kernel.
__global__ void __launch_bounds__(128) append_pages_kernel(const __grid_constant__ AppendParams p) {
  const int b = blockIdx.z, g = blockIdx.y, tid = threadIdx.x;
  const int n = p.seq_len[b];
  const int end = n + p.n_new;
  if (n < 0 || end > p.max_pages * p.P) {
    if (blockIdx.x == 0 && g == 0 && tid == 0) flag_error(p.err, RKV_DEVERR_CAPACITY);
    return;
  }
  const int pg = n / p.P + blockIdx.x;
  if (pg * p.P >= end) return;
  const int phys = p.page_table[(size_t)b * p.max_pages + pg];
  if (!phys_ok(p, phys)) return;
  if (p.k_new) {
    const int lo = max(n, pg * p.P), hi = min(end, (pg + 1) * p.P);
    const int c2 = tid & 63;
    for (int pos = lo + (tid >> 6); pos < hi; pos += 2) {
      const int i = pos - n;
      const size_t dst = (((size_t)phys * p.Hkv + g) * p.P + pos % p.P) * 128 + 2 * c2;
      const size_t src = (((size_t)b * p.Hkv + g) * p.n_new + i) * 128 + 2 * c2;
      *reinterpret_cast<uint32_t*>(p.k_pages + dst) = *reinterpret_cast<const uint32_t*>(p.k_new + src);
      *reinterpret_cast<uint32_t*>(p.v_pages + dst) = *reinterpret_cast<const uint32_t*>(p.v_new + src);
    }
    __syncthreads();
  }
  if (tid < 64) summarize_pair(p, b, g, pg, phys, min(p.P, end - pg * p.P), tid);
}

__global__ void append_advance_kernel(const __grid_constant__ AppendParams p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const int n = p.seq_len[b];
  if (n >= 0 && n + p.n_new <= p.max_pages * p.P) p.seq_len[b] = n + p.n_new;
}

}  // namespace

cudaError_t launch_append(const rkv_cache& c, const rkv_bf16* k_new, const rkv_bf16* v_new, int n_new,
                          cudaStream_t s) {
  AppendParams p;
  p.k_pages = c.k_pages;
  p.v_pages = c.v_pages;
  p.page_table = c.page_table;
  p.seq_len = c.seq_len;
  p.kmax = c.kmax;
  p.kmin = c.kmin;
  p.err = c.error_word;
  p.k_new = k_new;
  p.v_new = v_new;
  p.B = c.B;
  p.Hkv = c.Hkv;
  p.P = c.page_size;
  p.max_pages = c.max_pages;
  p.num_phys = c.num_phys_pages;
  p.n_new = n_new;
  if (n_new <= 16) {
    launch_begin(K_APPEND_SMALL, s);
    append_small_kernel<<<c.B, 256, 0, s>>>(p);
    launch_end(K_APPEND_SMALL, s);
  } else {
    const int pages = (n_new + c.page_size - 1) / c.page_size + 1;
    launch_begin(K_APPEND_PAGES, s);
    append_pages_kernel<<<dim3(pages, c.Hkv, c.B), 128, 0, s>>>(p);
    launch_end(K_APPEND_PAGES, s);
    launch_begin(K_APPEND_ADVANCE, s);
    append_advance_kernel<<<(c.B + 127) / 128, 128, 0, s>>>(p);
    launch_end(K_APPEND_ADVANCE, s);
  }
  return cudaGetLastError();
}

}  // namespace rkv
