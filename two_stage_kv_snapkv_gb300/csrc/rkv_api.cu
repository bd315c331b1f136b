// C ABI of librkv: argument validation, the adaptive ratio split, dispatch to the
// kernel launchers, error reporting, launch counting and optional per-kernel timing.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>
#include <atomic>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "rkv.h"
#include "rkv_internal.h"

namespace {

// An NVTX range over one library call, named after it: the calls show up on an Nsight
// timeline around their kernels.  Without a tool attached a push or pop is a no-op.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

thread_local std::string g_err;
std::atomic<long long> g_launches{0};
std::atomic<int> g_decode_path{0};

rkv_status fail(rkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rkv_status check_cache(const rkv_cache* c) {
  if (!c) return fail(RKV_ERR_INVALID_ARG, "cache is NULL");
  if (c->head_dim != RKV_HEAD_DIM) return fail(RKV_ERR_UNSUPPORTED, "head_dim %d unsupported (only 128)", c->head_dim);
  if (c->B < 1 || c->B > RKV_MAX_BATCH) return fail(RKV_ERR_INVALID_ARG, "B=%d outside [1, %d]", c->B, RKV_MAX_BATCH);
  if (c->Hkv < 1) return fail(RKV_ERR_INVALID_ARG, "Hkv=%d", c->Hkv);
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64)
    return fail(RKV_ERR_UNSUPPORTED, "page_size %d unsupported (16, 32 or 64)", c->page_size);
  if (c->max_pages < 8 || c->max_pages % 8 != 0)
    return fail(RKV_ERR_INVALID_ARG, "max_pages=%d must be a positive multiple of 8", c->max_pages);
  if (c->max_pages > 16384) return fail(RKV_ERR_UNSUPPORTED, "max_pages=%d above 16384", c->max_pages);
  if (c->num_phys_pages < 1) return fail(RKV_ERR_INVALID_ARG, "num_phys_pages=%d", c->num_phys_pages);
  if ((long long)c->num_phys_pages * c->Hkv * c->page_size >= (1LL << 31))
    return fail(RKV_ERR_UNSUPPORTED, "the page pools' rows are indexed with 32-bit integers (TMA coordinates)");
  if (!c->k_pages || !c->v_pages || !c->page_table || !c->seq_len || !c->kmax || !c->kmin || !c->error_word)
    return fail(RKV_ERR_INVALID_ARG, "a cache pointer is NULL");
  if (!al16(c->k_pages) || !al16(c->v_pages) || !al16(c->page_table) || !al16(c->kmax) || !al16(c->kmin))
    return fail(RKV_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  return RKV_OK;
}

rkv_status check_heads(int Hq, int Hkv) {
  if (Hq < 1 || Hq % Hkv != 0) return fail(RKV_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(RKV_ERR_UNSUPPORTED, "group size %d unsupported", G);
  return RKV_OK;
}

rkv_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return RKV_OK;
  return fail(RKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------------ profiling
struct Pending {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<cudaEvent_t> g_pool;
std::vector<Pending> g_pending;
cudaEvent_t g_open[rkv::K_NUM_KINDS];
long long g_count[rkv::K_NUM_KINDS];
double g_ms[rkv::K_NUM_KINDS];

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Adds the elapsed time of every recorded pair to the totals; the pairs stay
// recorded (a captured graph re-records the same events on every replay).
void accumulate_locked() {
  for (const Pending& p : g_pending) {
    cudaEventSynchronize(p.b);
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) ms = 0.f;
    g_count[p.kind] += 1;
    g_ms[p.kind] += ms;
  }
}

void release_locked() {
  for (const Pending& p : g_pending) {
    g_pool.push_back(p.a);
    g_pool.push_back(p.b);
  }
  g_pending.clear();
}

}  // namespace

namespace rkv {

const char* kernel_name(int kind) {
  static const char* names[K_NUM_KINDS] = {
      "append_small", "append_pages", "append_advance", "snap_stats",  "snap_stats_combine",
      "snap_colsum",  "snap_pool",    "snap_select",    "snap_compact", "hsa_score",
      "hsa_topk",     "hsa_attend",   "hsa_combine",    "hsa_step",     "recall",
      "chunk_gather", "sparq_score",  "sparq_topk",     "sparq_attend", "wait_selftest",
      "sparq_keys_sync"};
  return (kind >= 0 && kind < K_NUM_KINDS) ? names[kind] : nullptr;
}

// Inside a stream capture a plain record only orders the capture; the external
// flag makes it a timing node of the graph.
void record(cudaEvent_t e, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(stream, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, stream, cudaEventRecordExternal);
  else
    cudaEventRecord(e, stream);
}

void launch_begin(int kind, cudaStream_t stream) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t e = take_event();
  record(e, stream);
  g_open[kind] = e;
}

void launch_end(int kind, cudaStream_t stream) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_open[kind]) return;
  cudaEvent_t e = take_event();
  record(e, stream);
  g_pending.push_back({kind, g_open[kind], e});
  g_open[kind] = nullptr;
}

void set_last_error(const char* msg) { g_err = msg ? msg : ""; }

int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}


bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  // cuTensorMapEncodeTiled from the driver, looked up once per process
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!enc) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rkv

extern "C" {

rkv_status rkv_split_ratio(int32_t prompt_len, int32_t budget, int32_t head_dim, int32_t page_size, int32_t window,
                           int32_t k1_override, rkv_split* out) {
  if (!out) return fail(RKV_ERR_INVALID_ARG, "out is NULL");
  if (prompt_len < 1 || budget < 1 || head_dim < 1 || page_size < 1 || window < 0 || k1_override < 0)
    return fail(RKV_ERR_INVALID_ARG, "sizes must be positive");
  const double c = (double)prompt_len / (double)budget;
  double r = 0.2 + 0.06 * std::log2(c);
  r = r < 0.2 ? 0.2 : (r > 0.8 ? 0.8 : r);
  const double c1 = std::pow(c, r), c2 = std::pow(c, 1.0 - r);
  long long keep1 = (long long)std::floor((double)prompt_len / c1 + 0.5);
  long long lo = budget > window ? budget : window;
  keep1 = keep1 < lo ? lo : keep1;
  keep1 = keep1 > prompt_len ? prompt_len : keep1;
  int k1 = k1_override;
  if (k1 <= 0) {
    k1 = 16 * (int)std::floor((double)head_dim / (16.0 * std::sqrt(c2)) + 0.5);
    k1 = k1 < 16 ? 16 : (k1 > head_dim ? head_dim : k1);
  }
  int k2 = budget / page_size;
  k2 = k2 < 1 ? 1 : k2;
  out->c = c;
  out->r = r;
  out->c1 = c1;
  out->c2 = c2;
  out->keep1 = (int32_t)keep1;
  out->k1 = k1;
  out->k2 = k2;
  out->pool_kernel = prompt_len <= 8192 ? 7 : (prompt_len <= 49152 ? 31 : 63);
  return RKV_OK;
}

rkv_status rkv_split_ratio_mt(int32_t prompt_len, int32_t budget, int32_t head_dim, int32_t page_size,
                              int32_t k1_override, rkv_split* out) {
  if (!out) return fail(RKV_ERR_INVALID_ARG, "out is NULL");
  if (prompt_len < 1 || budget < 1 || head_dim < 1 || page_size < 1 || k1_override < 0)
    return fail(RKV_ERR_INVALID_ARG, "sizes must be positive");
  const double c = (double)prompt_len / (double)budget;
  int k1 = k1_override;
  if (k1 <= 0) {
    k1 = 16 * (int)std::floor((double)head_dim / (16.0 * std::sqrt(c)) + 0.5);
    k1 = k1 < 16 ? 16 : (k1 > head_dim ? head_dim : k1);
  }
  int k2 = budget / page_size;
  k2 = k2 < 1 ? 1 : k2;
  out->c = c;
  out->r = 0.0;
  out->c1 = 1.0;
  out->c2 = c;
  out->keep1 = prompt_len;
  out->k1 = k1;
  out->k2 = k2;
  out->pool_kernel = prompt_len <= 8192 ? 7 : (prompt_len <= 49152 ? 31 : 63);
  return RKV_OK;
}

size_t rkv_prefill_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t window, int32_t max_prompt_len) {
  if (B < 1 || Hkv < 1 || max_prompt_len < 1) return 0;
  return rkv::prefill_ws_bytes(B, Hq, Hkv, window, max_prompt_len);
}

// Device address of pinned host memory mapped into the device's address space, else null.
// True when p is known to be host memory (pinned or not); false for device or managed
// memory, and when the query itself fails (then the launch reports any fault).
static bool host_side(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

static const void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // unregistered memory: clear the sticky query error
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

rkv_status rkv_prefill_evict(const rkv_bf16* q_win, const rkv_bf16* k, const rkv_bf16* v, int32_t B, int32_t Hq,
                             int32_t window, int32_t max_prompt_len, const int32_t* prompt_len, const int32_t* keep1,
                             const int32_t* pool_kernel, float scale, const rkv_cache* cache, int32_t* kept_idx,
                             int32_t kept_stride, float* pooled_scores, void* workspace, size_t workspace_bytes,
                             void* stream) {
  const NvtxRange nvtx_range("rkv_prefill_evict");
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if ((st = check_heads(Hq, cache->Hkv)) != RKV_OK) return st;
  if (B != cache->B) return fail(RKV_ERR_INVALID_ARG, "B=%d differs from cache B=%d", B, cache->B);
  if (!q_win || !k || !v || !kept_idx || !prompt_len || !keep1 || !pool_kernel || !workspace)
    return fail(RKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!al16(q_win) || !al16(k) || !al16(v) || !al16(kept_idx) || !al16(workspace) ||
      (pooled_scores && !al16(pooled_scores)))
    return fail(RKV_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  const int G = Hq / cache->Hkv;
  if (window < 1 || G * window > 128)
    return fail(RKV_ERR_UNSUPPORTED, "window=%d: need 1 <= G*window <= 128 (G=%d)", window, G);
  if (max_prompt_len < 1) return fail(RKV_ERR_INVALID_ARG, "max_prompt_len=%d", max_prompt_len);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "scale must be positive");
  for (int b = 0; b < B; ++b) {
    const int L = prompt_len[b], kk = keep1[b], kp = pool_kernel[b];
    if (L < window || L > max_prompt_len)
      return fail(RKV_ERR_INVALID_ARG, "prompt_len[%d]=%d outside [window, max_prompt_len]", b, L);
    if (kk < window || kk > L) return fail(RKV_ERR_INVALID_ARG, "keep1[%d]=%d outside [window, prompt_len]", b, kk);
    if (kk > cache->max_pages * cache->page_size)
      return fail(RKV_ERR_INVALID_ARG, "keep1[%d]=%d exceeds the cache capacity", b, kk);
    if (kk > kept_stride) return fail(RKV_ERR_INVALID_ARG, "kept_stride=%d < keep1[%d]=%d", kept_stride, b, kk);
    if (kp < 1 || kp > 255 || kp % 2 == 0)
      return fail(RKV_ERR_INVALID_ARG, "pool_kernel[%d]=%d must be odd in [1, 255]", b, kp);
  }
  const size_t need = rkv::prefill_ws_bytes(B, Hq, cache->Hkv, window, max_prompt_len);
  if (workspace_bytes < need)
    return fail(RKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  rkv::PrefillArgs a;
  a.q_win = q_win;
  a.k = k;
  // pinned host V: the compaction reads the kept rows through the device mapping.  q_win
  // and k are read by the tensor engine and must be device memory.
  if (host_side(q_win) || host_side(k)) return fail(RKV_ERR_INVALID_ARG, "q_win and k must be device memory");
  const void* vmap = mapped_host(v);
  if (!vmap && host_side(v)) return fail(RKV_ERR_INVALID_ARG, "v is host memory that is not pinned and mapped");
  a.v = vmap ? static_cast<const rkv_bf16*>(vmap) : v;
  if (!al16(a.v)) return fail(RKV_ERR_INVALID_ARG, "v's device mapping must be 16-byte aligned");
  a.B = B;
  a.Hq = Hq;
  a.Hkv = cache->Hkv;
  a.G = G;
  a.w = window;
  a.Lmax = max_prompt_len;
  a.prompt_len = prompt_len;
  a.keep1 = keep1;
  a.pool_kernel = pool_kernel;
  a.scale = scale;
  a.cache = *cache;
  a.kept_idx = kept_idx;
  a.kept_stride = kept_stride;
  a.pooled_out = pooled_scores;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  return cuda_status(rkv::launch_prefill(a, static_cast<cudaStream_t>(stream)), "rkv_prefill_evict launch");
}

size_t rkv_prefill_chunk_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t window, int32_t max_total_len) {
  if (B < 1 || Hkv < 1 || max_total_len < 1) return 0;
  return rkv::prefill_chunk_ws_bytes(B, Hq, Hkv, window, max_total_len);
}

rkv_status rkv_prefill_chunk(const rkv_bf16* q_win, const rkv_bf16* k_chunk, const rkv_bf16* v_chunk, int32_t B,
                             int32_t Hq, int32_t window, int32_t chunk_max, const int32_t* chunk_len,
                             const int32_t* held_len, const int32_t* keep1, const int32_t* pool_kernel, float scale,
                             const rkv_cache* cache, int32_t* kept_idx, int32_t kept_stride, void* workspace,
                             size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("rkv_prefill_chunk");
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if ((st = check_heads(Hq, cache->Hkv)) != RKV_OK) return st;
  if (B != cache->B) return fail(RKV_ERR_INVALID_ARG, "B=%d differs from cache B=%d", B, cache->B);
  if (!q_win || !k_chunk || !v_chunk || !kept_idx || !chunk_len || !held_len || !keep1 || !pool_kernel || !workspace)
    return fail(RKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!al16(q_win) || !al16(k_chunk) || !al16(v_chunk) || !al16(kept_idx) || !al16(workspace))
    return fail(RKV_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  const int G = Hq / cache->Hkv;
  if (window < 1 || G * window > 128)
    return fail(RKV_ERR_UNSUPPORTED, "window=%d: need 1 <= G*window <= 128 (G=%d)", window, G);
  if (chunk_max < 1) return fail(RKV_ERR_INVALID_ARG, "chunk_max=%d", chunk_max);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "scale must be positive");
  const long long cap = (long long)cache->max_pages * cache->page_size;
  long long Lc = 1;
  for (int b = 0; b < B; ++b) {
    const int m = chunk_len[b], h = held_len[b], kk = keep1[b], kp = pool_kernel[b];
    if (m < window || m > chunk_max)
      return fail(RKV_ERR_INVALID_ARG, "chunk_len[%d]=%d outside [window, chunk_max]", b, m);
    if (h < 0 || h > cap) return fail(RKV_ERR_INVALID_ARG, "held_len[%d]=%d outside [0, cache capacity]", b, h);
    if (kk < window) return fail(RKV_ERR_INVALID_ARG, "keep1[%d]=%d below window", b, kk);
    const long long n = (long long)h + m, keep = kk < n ? kk : n;
    if (n > INT32_MAX / 2) return fail(RKV_ERR_INVALID_ARG, "held_len[%d] + chunk_len[%d] too large", b, b);
    if (keep > cap) return fail(RKV_ERR_INVALID_ARG, "keep1[%d]=%d exceeds the cache capacity", b, kk);
    if (keep > kept_stride) return fail(RKV_ERR_INVALID_ARG, "kept_stride=%d < %lld kept in sequence %d", kept_stride, keep, b);
    if (kp < 1 || kp > 255 || kp % 2 == 0)
      return fail(RKV_ERR_INVALID_ARG, "pool_kernel[%d]=%d must be odd in [1, 255]", b, kp);
    Lc = n > Lc ? n : Lc;
  }
  const size_t need = rkv::prefill_chunk_ws_bytes(B, Hq, cache->Hkv, window, (int)Lc);
  if (workspace_bytes < need)
    return fail(RKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  rkv::PrefillChunkArgs a;
  a.q_win = q_win;
  a.k_chunk = k_chunk;
  a.v_chunk = v_chunk;
  a.Hq = Hq;
  a.w = window;
  a.chunk_max = chunk_max;
  a.chunk_len = chunk_len;
  a.held_len = held_len;
  a.keep1 = keep1;
  a.pool_kernel = pool_kernel;
  a.scale = scale;
  a.cache = *cache;
  a.kept_idx = kept_idx;
  a.kept_stride = kept_stride;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  return cuda_status(rkv::launch_prefill_chunk(a, static_cast<cudaStream_t>(stream)), "rkv_prefill_chunk launch");
}

rkv_status rkv_append_page_summary(const rkv_cache* cache, const rkv_bf16* k_new, const rkv_bf16* v_new,
                                   int32_t n_new, void* stream) {
  const NvtxRange nvtx_range("rkv_append_page_summary");
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if (n_new < 1) return fail(RKV_ERR_INVALID_ARG, "n_new=%d", n_new);
  if (n_new > cache->max_pages * cache->page_size) return fail(RKV_ERR_INVALID_ARG, "n_new=%d exceeds capacity", n_new);
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(RKV_ERR_INVALID_ARG, "k_new and v_new must both be set");
  if (k_new && (!al16(k_new) || !al16(v_new))) return fail(RKV_ERR_INVALID_ARG, "k_new/v_new must be 16-byte aligned");
  return cuda_status(rkv::launch_append(*cache, k_new, v_new, n_new, static_cast<cudaStream_t>(stream)),
                     "rkv_append_page_summary launch");
}

size_t rkv_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_pages) {
  if (B < 1 || Hq < 1 || Hkv < 1 || max_pages < 1) return 0;
  return rkv::decode_ws_bytes(B, Hq, Hkv, max_pages);
}

static rkv_status decode_common(const rkv_cache* cache, const rkv_bf16* q, const rkv_bf16* k_new,
                                const rkv_bf16* v_new, int32_t Hq, const int32_t* k1, const int32_t* k2, float scale,
                                float* out, int32_t* sel_channels, int32_t* sel_pages, int32_t sel_pages_stride,
                                void* workspace, size_t workspace_bytes, void* stream, const char* who,
                                bool validate_only = false) {
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if ((st = check_heads(Hq, cache->Hkv)) != RKV_OK) return st;
  if (!q || !k1 || !k2 || !out || !workspace) return fail(RKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!al16(q) || !al16(out) || !al16(workspace) || (sel_channels && !al16(sel_channels)) ||
      (sel_pages && !al16(sel_pages)))
    return fail(RKV_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (k_new) {
    if (!v_new) return fail(RKV_ERR_INVALID_ARG, "k_new and v_new must both be set");
    if (!al16(k_new) || !al16(v_new)) return fail(RKV_ERR_INVALID_ARG, "k_new/v_new must be 16-byte aligned");
    if (!cache->step_sync) return fail(RKV_ERR_INVALID_ARG, "cache->step_sync is NULL");
  }
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "scale must be positive");
  for (int b = 0; b < cache->B; ++b) {
    if (k1[b] < 1 || k1[b] > RKV_HEAD_DIM) return fail(RKV_ERR_INVALID_ARG, "k1[%d]=%d outside [1, 128]", b, k1[b]);
    if (k2[b] < 1) return fail(RKV_ERR_INVALID_ARG, "k2[%d]=%d", b, k2[b]);
    if (sel_pages) {
      const int kk = k2[b] < cache->max_pages ? k2[b] : cache->max_pages;
      if (sel_pages_stride < kk) return fail(RKV_ERR_INVALID_ARG, "sel_pages_stride=%d < %d", sel_pages_stride, kk);
    }
  }
  const size_t need = rkv::decode_ws_bytes(cache->B, Hq, cache->Hkv, cache->max_pages);
  if (workspace_bytes < need)
    return fail(RKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (validate_only) return RKV_OK;
  rkv::DecodeArgs a;
  a.cache = *cache;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.mode = g_decode_path.load();
  a.Hq = Hq;
  a.G = Hq / cache->Hkv;
  a.k1 = k1;
  a.k2 = k2;
  a.scale = scale;
  a.out = out;
  a.sel_channels = sel_channels;
  a.sel_pages = sel_pages;
  a.sel_pages_stride = sel_pages_stride;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  return cuda_status(rkv::launch_decode(a, static_cast<cudaStream_t>(stream)), who);
}

rkv_status rkv_decode_hsa(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq, const int32_t* k1, const int32_t* k2,
                          float scale, float* out, int32_t* sel_channels, int32_t* sel_pages, int32_t sel_pages_stride,
                          void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("rkv_decode_hsa");
  return decode_common(cache, q, nullptr, nullptr, Hq, k1, k2, scale, out, sel_channels, sel_pages, sel_pages_stride,
                       workspace, workspace_bytes, stream, "rkv_decode_hsa launch");
}

rkv_status rkv_decode_step(const rkv_cache* cache, const rkv_bf16* q, const rkv_bf16* k_new, const rkv_bf16* v_new,
                           int32_t Hq, const int32_t* k1, const int32_t* k2, float scale, float* out,
                           int32_t* sel_channels, int32_t* sel_pages, int32_t sel_pages_stride, void* workspace,
                           size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("rkv_decode_step");
  if (!k_new || !v_new) return fail(RKV_ERR_INVALID_ARG, "rkv_decode_step needs k_new and v_new");
  return decode_common(cache, q, k_new, v_new, Hq, k1, k2, scale, out, sel_channels, sel_pages, sel_pages_stride,
                       workspace, workspace_bytes, stream, "rkv_decode_step launch");
}

size_t rkv_sparq_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_pages, int32_t page_size) {
  if (B < 1 || Hkv < 1 || max_pages < 1 || page_size < 1) return 0;
  return rkv::sparq_ws_bytes(B, Hq, Hkv, max_pages, page_size);
}

size_t rkv_sparq_keys_size(int32_t B, int32_t Hkv, int32_t max_pages, int32_t page_size) {
  if (B < 1 || Hkv < 1 || max_pages < 1 || page_size < 1) return 0;
  return rkv::sparq_keys_bytes(B, Hkv, max_pages, page_size);
}

rkv_status rkv_decode_sparq(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq, const int32_t* k1,
                            const int32_t* k_tokens, float scale, float* out, int32_t* sel_channels,
                            int32_t* sel_tokens, int32_t sel_tokens_stride, void* keys_t, size_t keys_t_bytes,
                            void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("rkv_decode_sparq");
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if ((st = check_heads(Hq, cache->Hkv)) != RKV_OK) return st;
  if (!q || !k1 || !k_tokens || !out || !workspace) return fail(RKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!al16(q) || !al16(out) || !al16(workspace) || (sel_channels && !al16(sel_channels)) ||
      (sel_tokens && !al16(sel_tokens)))
    return fail(RKV_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "scale must be positive");
  const long cap = (long)cache->max_pages * cache->page_size;
  if (cap > rkv::sparq_max_tokens())
    return fail(RKV_ERR_UNSUPPORTED, "the token path supports caches of at most %d tokens per sequence",
                rkv::sparq_max_tokens());
  for (int b = 0; b < cache->B; ++b) {
    if (k1[b] < 1 || k1[b] > RKV_HEAD_DIM) return fail(RKV_ERR_INVALID_ARG, "k1[%d]=%d outside [1, 128]", b, k1[b]);
    if (k_tokens[b] < 1) return fail(RKV_ERR_INVALID_ARG, "k_tokens[%d]=%d", b, k_tokens[b]);
    if (sel_tokens) {
      const long kk = k_tokens[b] < cap ? k_tokens[b] : cap;
      if (sel_tokens_stride < kk)
        return fail(RKV_ERR_INVALID_ARG, "sel_tokens_stride=%d < %ld", sel_tokens_stride, kk);
    }
  }
  const size_t need = rkv::sparq_ws_bytes(cache->B, Hq, cache->Hkv, cache->max_pages, cache->page_size);
  if (workspace_bytes < need)
    return fail(RKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (keys_t) {
    if (!al16(keys_t)) return fail(RKV_ERR_INVALID_ARG, "keys_t must be 16-byte aligned");
    const size_t kneed = rkv::sparq_keys_bytes(cache->B, cache->Hkv, cache->max_pages, cache->page_size);
    if (keys_t_bytes < kneed) return fail(RKV_ERR_WORKSPACE, "keys_t %zu bytes < %zu needed", keys_t_bytes, kneed);
  }
  rkv::DecodeArgs a;
  a.cache = *cache;
  a.q = q;
  a.k_new = nullptr;
  a.v_new = nullptr;
  a.mode = 0;
  a.Hq = Hq;
  a.G = Hq / cache->Hkv;
  a.k1 = k1;
  a.k2 = k_tokens;
  a.scale = scale;
  a.out = out;
  a.sel_channels = sel_channels;
  a.sel_pages = sel_tokens;
  a.sel_pages_stride = sel_tokens_stride;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.keys_t = keys_t;
  return cuda_status(rkv::launch_sparq(a, static_cast<cudaStream_t>(stream)), "rkv_decode_sparq launch");
}


size_t rkv_step_host_staging_size(int32_t B, int32_t Hq, int32_t Hkv) {
  if (B < 1 || Hq < 1 || Hkv < 1) return 0;
  const size_t in = (size_t)B * (Hq + 2 * Hkv) * RKV_HEAD_DIM * 2;
  return ((in + 255) & ~size_t(255)) + (size_t)B * Hq * RKV_HEAD_DIM * 4;
}

rkv_status rkv_decode_step_host(const rkv_cache* cache, const void* host_in, float* host_out, int32_t Hq,
                                const int32_t* k1, const int32_t* k2, float scale, void* staging,
                                size_t staging_bytes, void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("rkv_decode_step_host");
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if ((st = check_heads(Hq, cache->Hkv)) != RKV_OK) return st;
  if (!host_in || !host_out || !staging) return fail(RKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!al16(staging)) return fail(RKV_ERR_INVALID_ARG, "staging must be 16-byte aligned");
  const size_t need = rkv_step_host_staging_size(cache->B, Hq, cache->Hkv);
  if (staging_bytes < need) return fail(RKV_ERR_WORKSPACE, "staging %zu bytes < %zu needed", staging_bytes, need);
  const size_t nq = (size_t)cache->B * Hq * RKV_HEAD_DIM, nkv = (size_t)cache->B * cache->Hkv * RKV_HEAD_DIM;
  const size_t in_bytes = (nq + 2 * nkv) * 2;
  uint8_t* dev = static_cast<uint8_t*>(staging);
  const rkv_bf16* q = reinterpret_cast<const rkv_bf16*>(dev);
  const rkv_bf16* k_new = q + nq;
  const rkv_bf16* v_new = k_new + nkv;
  float* out = reinterpret_cast<float*>(dev + ((in_bytes + 255) & ~size_t(255)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // pinned host buffers mapped into the device's address space (all pinned memory is,
  // with unified addressing) are read and written by the kernel itself: no copies
  const void* din = mapped_host(host_in);
  void* dout = const_cast<void*>(mapped_host(host_out));
  if (din && dout && al16(din) && al16(dout)) {
    const rkv_bf16* hq = static_cast<const rkv_bf16*>(din);
    return decode_common(cache, hq, hq + nq, hq + nq + nkv, Hq, k1, k2, scale, static_cast<float*>(dout), nullptr,
                         nullptr, 0, workspace, workspace_bytes, stream, "rkv_decode_step_host launch");
  }
  // the step validates everything else before anything is enqueued
  st = decode_common(cache, q, k_new, v_new, Hq, k1, k2, scale, out, nullptr, nullptr, 0, workspace, workspace_bytes,
                     stream, "rkv_decode_step_host", true);
  if (st != RKV_OK) return st;
  cudaError_t e = cudaMemcpyAsync(dev, host_in, in_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_status(e, "rkv_decode_step_host input copy");
  st = decode_common(cache, q, k_new, v_new, Hq, k1, k2, scale, out, nullptr, nullptr, 0, workspace, workspace_bytes,
                     stream, "rkv_decode_step_host launch", false);
  if (st != RKV_OK) return st;
  e = cudaMemcpyAsync(host_out, out, (size_t)cache->B * Hq * RKV_HEAD_DIM * 4, cudaMemcpyDeviceToHost, s);
  return cuda_status(e, "rkv_decode_step_host output copy");
}

rkv_status rkv_exact_topk_recall(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq, const int32_t* sel_pages,
                                 int32_t sel_pages_stride, const int32_t* k_tokens, float scale, float* recall,
                                 float* mass, void* stream) {
  const NvtxRange nvtx_range("rkv_exact_topk_recall");
  rkv_status st = check_cache(cache);
  if (st != RKV_OK) return st;
  if ((st = check_heads(Hq, cache->Hkv)) != RKV_OK) return st;
  if (!q || !sel_pages || !k_tokens || !recall) return fail(RKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!al16(q) || !al16(recall) || (mass && !al16(mass)) || !al16(sel_pages))
    return fail(RKV_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (sel_pages_stride < 1) return fail(RKV_ERR_INVALID_ARG, "sel_pages_stride=%d", sel_pages_stride);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "scale must be positive");
  if ((long)cache->max_pages * cache->page_size > rkv::recall_max_tokens())
    return fail(RKV_ERR_UNSUPPORTED, "the recall diagnostic supports caches of at most %d tokens per sequence",
                rkv::recall_max_tokens());
  for (int b = 0; b < cache->B; ++b)
    if (k_tokens[b] < 0) return fail(RKV_ERR_INVALID_ARG, "k_tokens[%d]=%d", b, k_tokens[b]);
  rkv::RecallArgs a;
  a.cache = *cache;
  a.q = q;
  a.Hq = Hq;
  a.sel_pages = sel_pages;
  a.sel_pages_stride = sel_pages_stride;
  a.k_tokens = k_tokens;
  a.scale = scale;
  a.recall = recall;
  a.mass = mass;
  return cuda_status(rkv::launch_recall(a, static_cast<cudaStream_t>(stream)), "rkv_exact_topk_recall launch");
}

rkv_status rkv_selftest_bounded_wait(const rkv_cache* cache, int64_t limit_ns, void* stream) {
  const NvtxRange nvtx_range("rkv_selftest_bounded_wait");
  if (!cache || !cache->error_word) return fail(RKV_ERR_INVALID_ARG, "cache or error_word is NULL");
  if (reinterpret_cast<uintptr_t>(cache->error_word) & 3u)
    return fail(RKV_ERR_INVALID_ARG, "error_word must be 4-byte aligned");
  if (limit_ns < 1 || limit_ns > 1000000000LL)
    return fail(RKV_ERR_INVALID_ARG, "limit_ns=%lld must be in [1, 1e9]", (long long)limit_ns);
  return cuda_status(rkv::launch_wait_selftest(cache->error_word, (uint64_t)limit_ns, static_cast<cudaStream_t>(stream)),
                     "rkv_selftest_bounded_wait launch");
}

int32_t rkv_decode_path(int32_t path) {
  if (path >= 0 && path <= 2) g_decode_path.store(path);
  return g_decode_path.load();
}

rkv_status rkv_get_device_status(const rkv_cache* cache, void* stream, int32_t* bits) {
  const NvtxRange nvtx_range("rkv_get_device_status");
  if (!cache || !cache->error_word) return fail(RKV_ERR_INVALID_ARG, "cache or error_word is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, cache->error_word, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && word != 0) e = cudaMemsetAsync(cache->error_word, 0, sizeof word, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(RKV_ERR_CUDA, "rkv_get_device_status: %s", cudaGetErrorString(e));
  if (bits) *bits = word;
  if (word == 0) return RKV_OK;
  if (word & RKV_DEVERR_TIMEOUT) return fail(RKV_ERR_TIMEOUT, "a bounded device wait ran out (word 0x%x)", word);
  return fail(RKV_ERR_DEVICE_DATA, "device data error (word 0x%x)", word);
}

const char* rkv_last_error(void) { return g_err.c_str(); }

int64_t rkv_launch_count(void) { return (int64_t)g_launches.load(); }

void rkv_profile_enable(int32_t enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = enable != 0;
}

void rkv_profile_accumulate(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  accumulate_locked();
}

void rkv_profile_release(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  release_locked();
}

void rkv_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < rkv::K_NUM_KINDS; ++i) {
    g_count[i] = 0;
    g_ms[i] = 0.0;
  }
}

const char* rkv_profile_read(int32_t kind, int64_t* launches, double* total_ms) {
  if (kind < 0 || kind >= rkv::K_NUM_KINDS) return nullptr;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (launches) *launches = g_count[kind];
  if (total_ms) *total_ms = g_ms[kind];
  return rkv::kernel_name(kind);
}

}  // extern "C"
