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
constexpr unsigned kErrBadRecord = 4u; // the merge found no consistent split record

enum DType { F32 = 0, BF16 = 1 };

// ---------------------------------------------------------------------------
// Split-KV partition.
//
// Work is laid out on a cost axis: every valid sequence b (P_b = ceil(L_b/64)
// > 0 pages) covers C + P_b units, C units for the fixed cost of one work item
// (loading the query rows, the output epilogue) followed by one unit per page.
// With U units in all and W' = min(W, floor(U / (C + 1))) active workers (W
// launched), worker w < W' takes the units [floor(U*w/W'), floor(U*(w+1)/W'))
// and, of sequence b starting at unit A_b (its first page at A_b + C), the
// pages j with A_b + C + j in that range.  A worker whose range crosses into
// a new sequence so gets about C pages fewer, and the cost pages + C * items
// of the active workers differs by at most 2C + 1 units (a range holds the
// floor or ceiling of U / W' units; a worker starting inside a sequence's
// pages pays C for that item outside its units, and one whose range ends
// inside a sequence's C units holds units it does not pay for).  Each range
// spans at least C + 1
// units, so it holds at least one page and none is empty (the workers between
// a sequence's first and last one all hold a part of it).  With C = 0 this is
// the plain even split of the pages.  A sequence whose pages fall to a single
// worker is finished by that worker; otherwise every worker that touched it
// leaves a partial (o, lse) in slot b + w of the workspace (b + w is unique
// among intersecting (b, w) pairs because both ranges are ordered), and the
// combine kernel merges them.
// ---------------------------------------------------------------------------
__host__ __device__ inline int part_active(long long U, int W, int C) {
  const long long m = U / (long long)(C + 1);
  return (int)(m < (long long)W ? m : (long long)W);
}
// first unit of worker w
__host__ __device__ inline long long part_begin(long long U, int W, int w) {
  return (U * (long long)w) / W;
}
// the worker whose range holds unit x (0 <= x < U)
__host__ __device__ inline int part_worker_of(long long U, int W, long long x) {
  return (int)(((x + 1) * (long long)W - 1) / U);
}
// pages [*j0, *j1) of a sequence with P pages, the first at unit A, that lie
// in the units [x0, x1)
__host__ __device__ inline void part_pages(long long x0, long long x1, long long A, int P,
                                           int* j0, int* j1) {
  const long long a = x0 - A, b = x1 - A;
  *j0 = (int)(a < 0 ? 0 : a > P ? P : a);
  *j1 = (int)(b < 0 ? 0 : b > P ? P : b);
}

// Workspace layout for rows = T_q*H query rows per sequence, W split
// workers and msg_bytes of message ring per worker (the tensor-core kernel
// passes each page's probabilities from the score CTA to the value CTA
// through it; the CUDA-core kernel uses none).
struct WsLayout {
  size_t meta_off;   // int2 [B]: (first worker, last worker) of each sequence
  size_t lse_off;    // float [(B + W) * rows]
  size_t o_off;      // float [(B + W) * rows * d_c]
  size_t msg_off;    // W * msg_bytes
  size_t total;
};
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline WsLayout ws_layout(int B, int rows, int d_c, int W, size_t msg_bytes = 0) {
  WsLayout L;
  size_t slots = (size_t)B + (size_t)W;
  L.meta_off = 0;
  L.lse_off = align_up(sizeof(int) * 2 * (size_t)B, 256);
  L.o_off = align_up(L.lse_off + sizeof(float) * slots * rows, 256);
  L.msg_off = align_up(L.o_off + sizeof(float) * slots * rows * (size_t)d_c, 1024);
  L.total = align_up(L.msg_off + (size_t)W * msg_bytes, 256);
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
  unsigned char* msg;         // per-worker message rings (tensor-core kernel)
  int W;                      // number of split workers
  int item_cost;              // C of the split partition (units per work item)
  // Row groups: the tensor-core kernel handles at most 128 query rows of a
  // sequence at a time; a sequence with more rows is planned as G "virtual
  // sequences" (b, g), g < G, over the same pages, each with rows
  // [g * SR, min((g + 1) * SR, T_q * H)).  Workspace slots, partials and the
  // merge are per virtual sequence (b * G + g), SR rows each.  G = 1 and
  // SR = T_q * H otherwise.
  int G;
  int SR;
  unsigned* err;              // device error word
  // Test hook (zero in normal calls): when skip_load > 0 the tensor-core
  // kernel leaves out the shared-memory load of the skip_load-th page of
  // worker 0, so that the wait for it runs out after wait_ns and the call
  // reports MLA_ERR_TIMEOUT.
  int skip_load;
  unsigned long long wait_ns; // budget of every bounded wait (0: the default)
};

__device__ __forceinline__ float load_as_float(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

}  // namespace mla
