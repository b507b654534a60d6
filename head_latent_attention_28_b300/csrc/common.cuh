// Shared definitions of the MLA CUDA library (internal; not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mla {

constexpr int kPage = 64;  // tokens per cache block

// bits of the per-device error word
constexpr unsigned kErrBadIndex = 1u;  // block id or sequence length out of range
constexpr unsigned kErrTimeout = 2u;   // a bounded wait gave up

enum DType { F32 = 0, BF16 = 1 };

// ---------------------------------------------------------------------------
// Split-KV partition.
//
// Sequence b owns the global page range [S_b, S_b + P_b), P_b = ceil(L_b/64),
// S_b = sum_{b'<b} P_b'.  With T = sum_b P_b pages and W' = min(W, T) active
// workers (W launched), worker w < W' processes pages
// [floor(T*w/W'), floor(T*(w+1)/W')): every active worker gets the same
// number of pages give or take one, whatever the length mix, and none is
// empty (so the workers between a sequence's first and last one all hold a
// part of it).  A sequence
// whose pages fall to a single worker is finished by that worker; otherwise
// every worker that touched it leaves a partial (o, lse) in slot b + w of the
// workspace (b + w is unique among intersecting (b, w) pairs because both
// page ranges are ordered), and the combine kernel merges them.
// ---------------------------------------------------------------------------
__host__ __device__ inline int part_active(long long T, int W) {
  return (int)(T < (long long)W ? T : (long long)W);
}
__host__ __device__ inline long long part_begin(long long T, int W, int w) {
  return (T * (long long)w) / W;
}
// the worker whose range holds page p (0 <= p < T)
__host__ __device__ inline int part_worker_of(long long T, int W, long long p) {
  return (int)(((p + 1) * (long long)W - 1) / T);
}

// Workspace layout for rows = T_q*H query rows per sequence.
struct WsLayout {
  size_t meta_off;   // int2 [B]: (first worker, last worker) of each sequence
  size_t lse_off;    // float [(B + W) * rows]
  size_t o_off;      // float [(B + W) * rows * d_c]
  size_t total;
};
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline WsLayout ws_layout(int B, int rows, int d_c, int W) {
  WsLayout L;
  size_t slots = (size_t)B + (size_t)W;
  L.meta_off = 0;
  L.lse_off = align_up(sizeof(int) * 2 * (size_t)B, 256);
  L.o_off = align_up(L.lse_off + sizeof(float) * slots * rows, 256);
  L.total = align_up(L.o_off + sizeof(float) * slots * rows * (size_t)d_c, 256);
  return L;
}

// Arguments of one decode call after host validation.
struct DecodeArgs {
  const void* q;              // [B, T_q, H, D]
  const void* cache;          // [num_blocks, 64, D]
  const int32_t* block_table; // [B, max_blocks]
  const int32_t* seqlens;     // [B]
  int dtype;
  int B, T_q, H, d_c, d_r, D, max_blocks, num_blocks;
  float scale;                // softmax scale
  int causal;
  float* o;                   // [B, T_q, H, d_c]
  float* lse;                 // [B, T_q, H] or nullptr
  // workspace views
  int2* meta;
  float* ws_lse;
  float* ws_o;
  int W;                      // number of split workers
  unsigned* err;              // device error word
};

__device__ __forceinline__ float load_as_float(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

}  // namespace mla
