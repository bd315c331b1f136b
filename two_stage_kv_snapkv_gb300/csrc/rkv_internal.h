// Internal launcher interface between the C-ABI layer (rkv_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rkv.h"

namespace rkv {

// Kinds of kernel, for launch counting and the optional per-kernel timing.
enum KernelKind {
  K_APPEND_SMALL = 0,
  K_APPEND_PAGES,
  K_APPEND_ADVANCE,
  K_SNAP_STATS,
  K_SNAP_STATS_COMBINE,
  K_SNAP_COLSUM,
  K_SNAP_POOL,
  K_SNAP_SELECT,
  K_SNAP_COMPACT,
  K_HSA_SCORE,
  K_HSA_TOPK,
  K_HSA_ATTEND,
  K_HSA_COMBINE,
  K_HSA_STEP,
  K_RECALL,
  K_CHUNK_GATHER,
  K_SPARQ_SCORE,
  K_SPARQ_TOPK,
  K_SPARQ_ATTEND,
  K_WAIT_SELFTEST,
  K_SPARQ_KEYS_SYNC,
  K_NUM_KINDS
};
const char* kernel_name(int kind);

// Launch bookkeeping: counting and, when enabled, event brackets on `stream`.
void launch_begin(int kind, cudaStream_t stream);
void launch_end(int kind, cudaStream_t stream);
int num_sms();
// Sets the message rkv_last_error() returns on this thread.
void set_last_error(const char* msg);

// A [rows][128] bf16 array as a 2-D tensor map of box_rows x 64-element boxes with
// 128-byte swizzle (a box row is 128 B; its 16-byte pieces are XOR-ed with row % 8).
// False when the driver's encoder is unavailable or rejects the map.
bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);

// --------------------------------------------------------------- cache append
cudaError_t launch_append(const rkv_cache& c, const rkv_bf16* k_new, const rkv_bf16* v_new,
                          int n_new, cudaStream_t s);

// --------------------------------------------------------------- prefill
struct PrefillArgs {
  const rkv_bf16* q_win;
  const rkv_bf16* k;
  const rkv_bf16* v;
  int B, Hq, Hkv, G, w, Lmax;
  const int32_t* prompt_len;   // host [B]
  const int32_t* keep1;        // host [B]
  const int32_t* pool_kernel;  // host [B]
  float scale;
  rkv_cache cache;
  int32_t* kept_idx;
  int kept_stride;
  float* pooled_out;  // may be null
  void* ws;
  size_t ws_bytes;
};
size_t prefill_ws_bytes(int B, int Hq, int Hkv, int w, int Lmax);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);

// Chunked prefill: the held survivors plus one chunk, re-evicted to keep1.
struct PrefillChunkArgs {
  const rkv_bf16* q_win;    // [B][Hq][w][128]: the chunk's last w queries
  const rkv_bf16* k_chunk;  // [B][Hkv][chunk_max][128]
  const rkv_bf16* v_chunk;
  int Hq, w, chunk_max;
  const int32_t* chunk_len;   // host [B]
  const int32_t* held_len;    // host [B]
  const int32_t* keep1;       // host [B]
  const int32_t* pool_kernel; // host [B]
  float scale;
  rkv_cache cache;
  int32_t* kept_idx;
  int kept_stride;
  void* ws;
  size_t ws_bytes;
};
size_t prefill_chunk_ws_bytes(int B, int Hq, int Hkv, int w, int Lc);
cudaError_t launch_prefill_chunk(const PrefillChunkArgs& a, cudaStream_t s);

// --------------------------------------------------------------- decode
enum DecodePath { DECODE_AUTO = 0, DECODE_SPLIT = 1, DECODE_FUSED = 2 };
struct DecodeArgs {
  rkv_cache cache;
  const rkv_bf16* q;
  const rkv_bf16* k_new;  // null: no append (rkv_decode_hsa)
  const rkv_bf16* v_new;
  int mode;               // DecodePath
  int Hq, G;
  const int32_t* k1;  // host [B]
  const int32_t* k2;  // host [B]
  float scale;
  float* out;
  int32_t* sel_channels;
  int32_t* sel_pages;
  int sel_pages_stride;
  void* ws;
  size_t ws_bytes;
  void* keys_t = nullptr;  // token path: the channel-major key copy, or null
};
size_t decode_ws_bytes(int B, int Hq, int Hkv, int max_pages);
// Token path (SparQ-only): k2 counts tokens; k_new must be null.
size_t sparq_ws_bytes(int B, int Hq, int Hkv, int max_pages, int page_size);
int sparq_max_tokens();
size_t sparq_keys_bytes(int B, int Hkv, int max_pages, int page_size);
cudaError_t launch_sparq(const DecodeArgs& a, cudaStream_t s);
bool decode_fused_ok(const rkv_cache& c);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// --------------------------------------------------------------- diagnostics
struct RecallArgs {
  rkv_cache cache;
  const rkv_bf16* q;
  int Hq;
  const int32_t* sel_pages;
  int sel_pages_stride;
  const int32_t* k_tokens;  // host [B]
  float scale;
  float* recall;
  float* mass;  // may be null
};
int recall_max_tokens();
cudaError_t launch_recall(const RecallArgs& a, cudaStream_t s);

// One CTA that waits, for at most limit_ns, on an mbarrier nothing arrives on, and
// flags RKV_DEVERR_TIMEOUT in err when the wait runs out (the failure path's test).
cudaError_t launch_wait_selftest(int32_t* err, uint64_t limit_ns, cudaStream_t s);

}  // namespace rkv
