// Prefill with materialised per-head keys and values (bf16, d_c = 512,
// d_h = 128, d^R_h = 64).
//
// For a chunk of T new tokens the absorbed path costs 2 (d_c + d^R_h) +
// 2 d_c flops per (query, key, head) pair; rebuilding every head's content
// key k_{s,h} = W^UK_h c_s and value v_{s,h} = W^UV_h c_s once per cached row
// ("Attention, Part 2: MQA, GQA and MLA", the MLA equations: the key of head
// h is [W^UK_h c_s ; R_s k^R_s], its value W^UV_h c_s) brings that down to
// 2 (d_h + d^R_h) + 2 d_h, plus 4 d_c d_h per (row, head) for the rebuild.
// Past a few dozen new tokens, attention over the rebuilt keys is the cheaper
// way ("Multi-head latent attention (MLA)", section 2: the up-projections may
// be applied to the cached latent or absorbed; the result is the same).
//
// Two kernels:
//  * prefill_kv_kernel: one CTA per (sequence, 128-row tile, group of 8
//    heads).  TMA brings the tile's two cache pages (latent columns only,
//    128 x 512, kept for all heads of the group) and streams [W^UK_h ; W^UV_h]
//    (256 x 512) in 64-column chunks; tcgen05.mma with M = 128 rows, N = 256,
//    K = 512 accumulates both products of a head in TMEM (two buffers, so the
//    epilogue of one head overlaps the MMAs of the next).  Four warps convert
//    to bf16 and write k_nope[b, h, s, :] and v[b, h, s, :]; rows past the
//    sequence end inside its last tile are written as zeros.  The first head
//    group also copies the rotated rotary key R_s k^R_s of each row.  For a
//    chunk of a chunked prefill only the chunk's rows [L - T_new, L) are
//    written (tiles below them exit at once); earlier rows stay as the
//    earlier chunks wrote them.
//  * prefill_attn_kernel: persistent, one CTA per SM, each taking work items
//    (a 128-token query tile of one head of one sequence; the items of a
//    head one after another, latest query tile first) from a counter until
//    none are left.  Scores over d_h + d^R_h = 192 dims (M = 128 queries,
//    N = 128 keys) go into one of two TMEM buffers.  Two groups of four
//    softmax warps split every key tile in halves of 64 keys; each half runs
//    its own base-2 online softmax with a lazy running max (its output is
//    rescaled only when a row maximum grows by more than 2^8; exact after the
//    final division), writes its bf16 probabilities over its own scores in
//    TMEM and accumulates O_h += P_h . V_h in its own TMEM accumulator (P read
//    from TMEM as the tcgen05.mma A operand).  The halves merge once, at the
//    end.  Key and value tiles stream through two-stage rings that run on
//    from one item into the next, so the scores of tile j + 1 run while the
//    softmax of tile j does, and the next item's first tiles load while the
//    current one finishes.  The query's rotary half is copied unrotated and
//    rotated in place (the same fixed-point angle table as the query
//    absorption).  Outputs leave through a small per-warp buffer so that each
//    store instruction writes 16 rows x 32 contiguous bytes.
// Every mbarrier wait is bounded (2 s): on expiry the kernel records
// MLA_ERR_TIMEOUT, lets its copies and MMAs finish, frees TMEM and returns.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int kPfThreads = 192;          // 6 warps: producer, MMA issuer, 4 row warps
constexpr int kBox16 = 16384;            // 128 rows x 64 dims bf16 (one SW128 box)
constexpr uint64_t kPfWaitNs = 2000000000ull;
constexpr float kPfLog2e = 1.4426950408889634f;
constexpr float kPfLn2 = 0.6931471805599453f;
constexpr float kPfRescale = 8.0f;       // lazy rescale threshold (log2 units)

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// every thread of the warp agrees that the wait succeeded; else the CTA aborts
__device__ __forceinline__ bool warp_ok(bool ok, volatile int* abort_flag, unsigned* err) {
  const bool all = __all_sync(0xffffffffu, ok);
  if (!all && (threadIdx.x & 31) == 0) {
    *abort_flag = 1;
    atomicOr(err, kErrTimeout);
  }
  return all;
}

// ---------------------------------------------------------------------------
// K/V rebuild
// ---------------------------------------------------------------------------
constexpr int kKvHeads = 8;              // heads per CTA (the latent tile is reused)
constexpr int kKvStages = 2;             // weight chunk ring
constexpr int kKvA = 8 * kBox16;         // 128 rows x 512 latents
constexpr int kKvW = 2 * kBox16;         // 64-column chunk of W^UK_h (128 rows) and W^UV_h (128 rows)
constexpr int kKvSmem = kKvA + kKvStages * kKvW + 1024;

__global__ void __launch_bounds__(kPfThreads, 1)
prefill_kv_kernel(const PrefillKvArgs a, const __grid_constant__ CUtensorMap tm_pool,
                  const __grid_constant__ CUtensorMap tm_wuk, const __grid_constant__ CUtensorMap tm_wuv) {
  extern __shared__ uint8_t kv_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(kv_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t a_full, w_full[kKvStages], w_empty[kKvStages], d_full[2], d_empty[2], mma_final;
  __shared__ uint32_t tbase;
  __shared__ int abort_raw, never_raw;
  volatile int* abort_flag = &abort_raw;
  volatile int* never = &never_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * kKvHeads;
  const int nh = min(kKvHeads, a.H - h0);
  const int L = a.seqlens[b];
  if (L < 0 || L > a.max_blocks * kPage) {
    if (threadIdx.x == 0 && tile == 0 && blockIdx.z == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const int r0 = tile * 128;
  if (r0 >= L) return;   // the whole CTA: no row of this sequence here
  // a chunk's rebuild writes only the new rows [L - T_new, L) (earlier rows
  // are the caller's from earlier chunks)
  const int row_lo = a.T_new > 0 ? max(0, L - a.T_new) : 0;
  if (r0 + 128 <= row_lo) return;
  const int pages = (L + kPage - 1) / kPage;

  if (threadIdx.x == 0) {
    abort_raw = 0;
    never_raw = 0;
    mbar_init(&a_full, 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&d_full[d], 1);
      mbar_init(&d_empty[d], 4);
    }
    mbar_init(&mma_final, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 1) tmem_alloc(&tbase, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  uint8_t* sA = smem;
  uint8_t* sW = smem + kKvA;
  uint32_t n_issued = 0;   // producer: weight chunks issued

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_first();   // each latent tile is read by 16 CTAs at most
      const uint64_t pol_w = policy_evict_last();    // the weights are read by every tile
      int y[2];
      for (int p = 0; p < 2; ++p) {
        const int j = 2 * tile + p;
        int blk = -1;
        if (j < pages) blk = a.block_table[(size_t)b * a.max_blocks + j];
        const bool ok = blk >= 0 && blk < a.num_blocks;
        if (j < pages && !ok) atomicOr(a.err, kErrBadIndex);
        // a page past the sequence (or an invalid one) reads past the pool's end: zeros
        y[p] = ok ? blk * kPage : a.num_blocks * kPage;
      }
      mbar_arrive_expect_tx(&a_full, kKvA);
      for (int c = 0; c < 8; ++c)
        for (int p = 0; p < 2; ++p)
          tma_load_2d(sA + c * kBox16 + p * 8192, &tm_pool, &a_full, 64 * c, y[p], pol_a);
      for (int hh = 0; hh < nh; ++hh) {
        const int wrow = (h0 + hh) * a.d_h;
        for (int c = 0; c < 8; ++c) {
          const uint32_t g = n_issued, s = g % kKvStages;
          if (g >= (uint32_t)kKvStages &&
              !mbar_wait(&w_empty[s], ((g / kKvStages) - 1) & 1, abort_flag, kPfWaitNs)) {
            *abort_flag = 1;
            atomicOr(a.err, kErrTimeout);
            break;
          }
          uint8_t* dst = sW + s * kKvW;
          mbar_arrive_expect_tx(&w_full[s], kKvW);
          tma_load_2d(dst, &tm_wuk, &w_full[s], 64 * c, wrow, pol_w);
          tma_load_2d(dst + kBox16, &tm_wuv, &w_full[s], 64 * c, wrow, pol_w);
          ++n_issued;
        }
        if (*abort_flag) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(128, 256, 0, 0);   // A and B K-major
      bool ok = mbar_wait(&a_full, 0, abort_flag, kPfWaitNs);
      uint32_t g = 0;
      for (int hh = 0; ok && hh < nh; ++hh) {
        const uint32_t d = hh & 1;
        if (hh >= 2) ok = mbar_wait(&d_empty[d], ((hh >> 1) - 1) & 1, abort_flag, kPfWaitNs);
        for (int c = 0; ok && c < 8; ++c, ++g) {
          const uint32_t s = g % kKvStages;
          ok = mbar_wait(&w_full[s], (g / kKvStages) & 1, abort_flag, kPfWaitNs);
          if (!ok) break;
          tc_fence_after();
          const uint8_t* wb = sW + s * kKvW;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint64_t ad = sdesc_sw128(smem_u32(sA + c * kBox16 + q * 32), 16, 1024);
            const uint64_t bd = sdesc_sw128(smem_u32(wb + q * 32), 16, 1024);
            mma_ss(tmem + d * 256, ad, bd, id, (c > 0 || q > 0) ? 1 : 0);
          }
          mma_commit(&w_empty[s]);
        }
        if (ok) mma_commit(&d_full[d]);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else {
    // row warps: TMEM lane quarter warp & 3 holds rows 32 (warp & 3) .. + 31
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int row = r0 + r;
    const bool real = row < L;
    const bool mine = row >= row_lo;   // rows of earlier chunks are left as they are
    const size_t orow = (size_t)b * a.R + row;
    if (blockIdx.z == 0 && mine) {
      // R_s k^R_s, unchanged from the cache row (zeros past the sequence end)
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.k_rope) + orow * a.d_r);
      int blk = -1;
      if (real) blk = a.block_table[(size_t)b * a.max_blocks + row / kPage];
      if (real && blk >= 0 && blk < a.num_blocks) {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(a.cache) +
            ((size_t)blk * kPage + row % kPage) * (a.d_c + a.d_r) + a.d_c);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = __ldg(src + k);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    for (int hh = 0; hh < nh; ++hh) {
      const uint32_t d = hh & 1;
      if (!warp_ok(mbar_wait(&d_full[d], (hh >> 1) & 1, abort_flag, kPfWaitNs), abort_flag, a.err))
        break;
      tc_fence_after();
      const size_t off = (((size_t)b * a.H + (h0 + hh)) * a.R + row) * a.d_h;
      __nv_bfloat16* kd = static_cast<__nv_bfloat16*>(a.k_nope) + off;
      __nv_bfloat16* vd = static_cast<__nv_bfloat16*>(a.v) + off;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float x[32];
        tmem_ld32(tmem + lane_off + d * 256 + 32 * c, x);
        tmem_ld_wait();
        uint4* dst = reinterpret_cast<uint4*>((c < 4 ? kd : vd) + 32 * (c & 3));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (real)
            w = make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]), pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                           pack_bf16x2(x[8 * i + 4], x[8 * i + 5]), pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
          if (mine) dst[i] = w;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[d]);
    }
  }

  // ---- drain: MMAs complete, copies landed, then free TMEM
  __syncwarp();
  if (warp == 1 && lane == 0) {
    mma_commit(&mma_final);
    if (!mbar_wait(&mma_final, 0, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
  }
  if (warp == 0 && lane == 0) {
    if (!mbar_wait(&a_full, 0, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
    for (uint32_t k = 0; k < (uint32_t)kKvStages && k < n_issued; ++k) {
      const uint32_t g = n_issued - 1 - k;
      if (!mbar_wait(&w_full[g % kKvStages], (g / kKvStages) & 1, never, kPfWaitNs))
        atomicOr(a.err, kErrTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// attention over the rebuilt keys and values
// ---------------------------------------------------------------------------
constexpr int kAtQ = 3 * kBox16;         // query tile: q_nope (2 boxes), rotated q_rope (1 box)
constexpr int kAtK = 3 * kBox16;         // key tile: k_nope (2 boxes), k_rope (1 box)
constexpr int kAtV = 2 * kBox16;         // value tile
constexpr int kAtStages = 2;
constexpr int kAtOffK = kAtQ;
constexpr int kAtOffV = kAtOffK + kAtStages * kAtK;
constexpr int kAtOffE = kAtOffV + kAtStages * kAtV;   // per-warp output transpose buffers
constexpr int kAtEpi = 1024;             // 32 rows x 8 fp32 per row warp
constexpr int kAtSmem = kAtOffE + 8 * kAtEpi + 1024;
constexpr int kAtThreads = 320;          // 10 warps: producer, MMA issuer, 2 x 4 row warps
// TMEM columns: two score buffers (each half's probabilities overwrite the
// first 32 columns of its half of the buffer), then the two halves' outputs
constexpr uint32_t kTS = 0, kTO = 256;
constexpr int kAtSlots = 64;             // work counters: one per stream that launches the kernel

// work counters of the persistent attention kernel: [0] next item, [1] CTAs
// finished (the last CTA to finish zeroes both for the next launch)
__device__ unsigned g_at_work[kAtSlots][2];

// a work item: one 128-token query tile of one head of one sequence.  Items
// are numbered head by head (so the CTAs running at any time share the keys
// and values of a few heads in L2), latest query tile first within a head
// (it sees the most keys).
struct AtItem {
  int qt, h, b;
};
__device__ __forceinline__ AtItem at_item(int i, int n_qt, int H) {
  const int hb = i / n_qt;
  return AtItem{n_qt - 1 - (i - hb * n_qt), hb % H, hb / H};
}
// key tiles a query tile sees (0 for a sequence of invalid length): keys 0 ..
// position of the tile's last query
__device__ __forceinline__ int at_key_tiles(const PrefillAttnArgs& a, const AtItem& it) {
  const int L = a.seqlens[it.b];
  if (L < a.T_q || L > a.max_len) return 0;
  const int last_t = min(it.qt * 128 + 127, a.T_q - 1);
  return (L - a.T_q + last_t) / 128 + 1;
}

// Persistent: each CTA takes work items (from a counter when `slot` >= 0, else
// items blockIdx.x, blockIdx.x + gridDim.x, ...) until none are left.  The
// producer publishes each item to the other roles through a two-entry ring.
// Key and value tiles stream through two-stage rings that run on from one item
// into the next; the next item's query tile is loaded as soon as the last
// score MMA of the current one has read the old one, and it is rotated by the
// row warps between the current item's last softmax and its output stores, so
// that the next item's first score MMAs overlap those stores.  The first value
// MMAs of an item wait until the row warps have read the previous item's
// outputs out of TMEM.
__global__ void __launch_bounds__(kAtThreads, 1)
prefill_attn_kernel(const PrefillAttnArgs a, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ RopeFreqs fr, int slot, int n_items) {
  extern __shared__ uint8_t at_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t q_full, q_ready, q_free, k_full[kAtStages], k_empty[kAtStages], v_full[kAtStages],
      v_empty[kAtStages], s_full[2], p_full[2], pv_done[2], grp, o_free, mma_final, item_full[2],
      item_empty[2];
  __shared__ float row_m[2][128], row_l[2][128];   // per-half row statistics for the final merge
  __shared__ int item_id[2];
  __shared__ uint32_t tbase;
  __shared__ int abort_raw, never_raw;
  volatile int* abort_flag = &abort_raw;
  volatile int* never = &never_raw;
  volatile int* items = item_id;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (a.T_q + 127) / 128;

  if (threadIdx.x == 0) {
    abort_raw = 0;
    never_raw = 0;
    mbar_init(&q_full, 1);
    mbar_init(&q_ready, 8);
    mbar_init(&q_free, 1);
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 8);
      mbar_init(&pv_done[s], 1);
      mbar_init(&item_full[s], 1);
      mbar_init(&item_empty[s], 9);   // the MMA issuer and the 8 row warps
    }
    mbar_init(&grp, 8);
    mbar_init(&o_free, 8);
    mbar_init(&mma_final, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 1) tmem_alloc(&tbase, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kAtOffK;
  uint8_t* sV = smem + kAtOffV;
  uint32_t n_k = 0, n_v = 0, n_q = 0;          // producer: key, value and query tiles issued

  // item n of this CTA, as published by the producer (-1: no more work)
  const auto fetch = [&](uint32_t n, int* out) -> bool {
    if (!mbar_wait(&item_full[n & 1], (n >> 1) & 1, abort_flag, kPfWaitNs)) return false;
    *out = items[n & 1];
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();   // every query tile of the head re-reads them
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        int i = slot >= 0 ? (int)atomicAdd(&g_at_work[slot][0], 1u) : (int)(blockIdx.x + n * gridDim.x);
        if (i >= n_items) i = -1;
        if (n >= 2 && !mbar_wait(&item_empty[n & 1], ((n >> 1) - 1) & 1, abort_flag, kPfWaitNs)) {
          ok = false;
          break;
        }
        items[n & 1] = i;
        mbar_arrive(&item_full[n & 1]);
        if (i < 0) break;
        const AtItem it = at_item(i, n_qt, a.H);
        const int n_kt = at_key_tiles(a, it);
        const int krow0 = (it.b * a.H + it.h) * a.R;   // first row of (sequence, head) in k_nope and v
        const int rrow0 = it.b * a.R;                  // first row of the sequence in k_rope
        const int n_tok = it.b * a.T_q + it.qt * 128;  // the tile's first query row in q_nope
        for (int j = 0; ok && j < n_kt; ++j) {
          const uint32_t s = n_k & 1;
          ok = n_k < 2 || mbar_wait(&k_empty[s], ((n_k >> 1) - 1) & 1, abort_flag, kPfWaitNs);
          if (!ok) break;
          uint8_t* kd = sK + s * kAtK;
          mbar_arrive_expect_tx(&k_full[s], kAtK);
          tma_load_3d(kd, &tm_k, &k_full[s], 0, krow0 + 128 * j, 0, pol_kv);   // both 64-dim halves
          tma_load_2d(kd + 2 * kBox16, &tm_kr, &k_full[s], 0, rrow0 + 128 * j, pol_kv);
          ++n_k;
          if (j == 0) {
            // the query tile, once the last score MMA of the previous item has read the old one
            ok = n_q == 0 || mbar_wait(&q_free, (n_q - 1) & 1, abort_flag, kPfWaitNs);
            if (!ok) break;
            mbar_arrive_expect_tx(&q_full, 3 * kBox16);
            tma_load_3d(sQ, &tm_q, &q_full, 0, it.h, n_tok, pol_q);
            tma_load_3d(sQ + kBox16, &tm_q, &q_full, 64, it.h, n_tok, pol_q);
            tma_load_3d(sQ + 2 * kBox16, &tm_qr, &q_full, 0, it.h, n_tok, pol_q);   // rotated in place
            ++n_q;
          }
          const uint32_t sv = n_v & 1;
          ok = n_v < 2 || mbar_wait(&v_empty[sv], ((n_v >> 1) - 1) & 1, abort_flag, kPfWaitNs);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full[sv], kAtV);
          tma_load_3d(sV + sv * kAtV, &tm_v, &v_full[sv], 0, krow0 + 128 * j, 0, pol_kv);
          ++n_v;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMAs issued by one thread run in issue order: the scores of tile
      // g + 2 overwrite the buffer that holds the probabilities of tile g only
      // after the value MMAs of tile g (issued earlier) have read them
      const uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);   // Q, K both K-major
      const uint32_t idO = idesc_bf16_f32(128, 128, 0, 1);   // P from TMEM, V MN-major
      bool ok = true;
      uint32_t g0 = 0, nq = 0;                 // key tiles and query tiles consumed
      for (uint32_t n = 0; ok; ++n) {
        int i;
        ok = fetch(n, &i);
        if (!ok) break;
        mbar_arrive(&item_empty[n & 1]);
        if (i < 0) break;
        const int n_kt = at_key_tiles(a, at_item(i, n_qt, a.H));
        if (n_kt == 0) continue;
        ok = mbar_wait(&q_full, nq & 1, abort_flag, kPfWaitNs) &&
             mbar_wait(&q_ready, nq & 1, abort_flag, kPfWaitNs);
        for (int j = 0; ok && j <= n_kt; ++j) {
          if (j < n_kt) {
            const uint32_t g = g0 + j, s = g & 1;
            ok = mbar_wait(&k_full[s], (g >> 1) & 1, abort_flag, kPfWaitNs);
            if (!ok) break;
            tc_fence_after();
            const uint8_t* kd = sK + s * kAtK;
#pragma unroll
            for (int kk = 0; kk < 12; ++kk) {
              const uint64_t ad = sdesc_sw128(smem_u32(sQ + (kk >> 2) * kBox16 + (kk & 3) * 32), 16, 1024);
              const uint64_t bd = sdesc_sw128(smem_u32(kd + (kk >> 2) * kBox16 + (kk & 3) * 32), 16, 1024);
              mma_ss(tmem + kTS + s * 128, ad, bd, idS, kk > 0 ? 1 : 0);
            }
            mma_commit(&k_empty[s]);
            mma_commit(&s_full[s]);
            if (j == n_kt - 1) mma_commit(&q_free);
          }
          if (j >= 1) {
            const uint32_t g = g0 + j - 1, s = g & 1;
            ok = mbar_wait(&p_full[s], (g >> 1) & 1, abort_flag, kPfWaitNs) &&
                 mbar_wait(&v_full[s], (g >> 1) & 1, abort_flag, kPfWaitNs);
            // the first value MMAs of an item overwrite the outputs: the row
            // warps must have read the previous item's
            if (ok && j == 1 && nq > 0) ok = mbar_wait(&o_free, (nq - 1) & 1, abort_flag, kPfWaitNs);
            if (!ok) break;
            tc_fence_after();
            const uint8_t* vd = sV + s * kAtV;
            // half hf: keys 64 hf .. 64 hf + 63 of the tile, its probabilities in
            // the first 32 columns of its half of the score buffer, into O_hf
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {   // 16 keys per step
                const uint64_t bd = sdesc_sw128(smem_u32(vd + (4 * hf + k4) * 2048), kBox16, 1024);
                mma_ts(tmem + kTO + hf * 128, tmem + kTS + s * 128 + hf * 64 + k4 * 8, bd, idO,
                       (j > 1 || k4 > 0) ? 1 : 0);
              }
            mma_commit(&v_empty[s]);
            mma_commit(&pv_done[s]);
          }
        }
        g0 += n_kt;
        ++nq;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else {
    // row warps: half hf (warps 2-5: keys 0-63 of every tile, warps 6-9: keys
    // 64-127) runs its own online softmax over its keys into its own output
    // accumulator O_hf; thread = query row r (TMEM lane r)
    const int hf = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float sl2 = a.scale * kPfLog2e;
    uint8_t* ebuf = smem + kAtOffE + (4 * hf + q4) * kAtEpi;
    uint32_t g0 = 0, nq = 0;                   // key tiles and query tiles consumed
    bool ok = true;

    // the query's rotary half was copied unrotated into box 2 of the query
    // tile (K-major, 128-byte swizzle: 16-byte chunk c of row r sits at chunk
    // c ^ (r & 7)); rotate it in place by the query's position, half hf taking
    // chunks 4 hf .. 4 hf + 3; rows past the sequence become zeros
    const auto rotate = [&](const AtItem& it, uint32_t q_index) -> bool {
      if (!warp_ok(mbar_wait(&q_full, q_index & 1, abort_flag, kPfWaitNs), abort_flag, a.err)) return false;
      const int t = it.qt * 128 + r;
      const int L = a.seqlens[it.b];
      const bool real = t < a.T_q;
      const uint64_t pos = (uint64_t)(int64_t)(L - a.T_q + t);
      uint8_t* qrow_s = sQ + 2 * kBox16 + r * 128;
#pragma unroll
      for (int c = 4 * hf; c < 4 * hf + 4; ++c) {   // 16-byte chunk c: rotary pairs 4c .. 4c + 3
        uint4* sl = reinterpret_cast<uint4*>(qrow_s + ((c ^ (r & 7)) << 4));
        const uint4 raw = *sl;
        const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (real) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * c + e;
            const float half_turns = (float)(int64_t)(pos * fr.turn[j]) * 0x1p-63f;
            float sn, cs;
            sincospif(half_turns, &sn, &cs);
            const float x1 = __uint_as_float(in[e] << 16), x2 = __uint_as_float(in[e] & 0xffff0000u);
            w[e] = pack_bf16x2(x1 * cs - x2 * sn, x1 * sn + x2 * cs);
          }
        }
        *sl = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_ready);
      return true;
    };

    uint32_t n = 0;
    int cur;
    ok = warp_ok(fetch(n, &cur), abort_flag, a.err);
    if (ok) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[n & 1]);
    }
    AtItem it{};
    int n_kt = 0;
    if (ok && cur >= 0) {
      it = at_item(cur, n_qt, a.H);
      n_kt = at_key_tiles(a, it);
      if (n_kt > 0) ok = rotate(it, nq);
    }
    while (ok && cur >= 0) {
      const int t = it.qt * 128 + r;
      const int L = a.seqlens[it.b];
      const size_t qrow = (size_t)it.b * a.T_q + t;
      float* orow = a.o + (qrow * a.H + it.h) * a.d_h;
      if (n_kt == 0) {
        // a sequence of invalid length: zeros (the error word says why)
        if (it.qt == 0 && it.h == 0 && lane == 0 && hf == 0 && q4 == 0) atomicOr(a.err, kErrBadIndex);
        if (t < a.T_q) {
          for (int c = 0; c < 16; ++c)
            reinterpret_cast<float4*>(orow + 64 * hf)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (hf == 0 && a.lse) a.lse[qrow * a.H + it.h] = 0.f;
        }
      } else {
        const int lim = t < a.T_q ? L - a.T_q + t : -1;   // position of the query = its last visible key
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; ok && j < n_kt; ++j) {
          const uint32_t g = g0 + j, s = g & 1;
          ok = warp_ok(mbar_wait(&s_full[s], (g >> 1) & 1, abort_flag, kPfWaitNs), abort_flag, a.err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sbuf = tmem + lane_off + kTS + s * 128 + hf * 64;
          float x[64];
          tmem_ld64(sbuf, x);
          tmem_ld_wait();
          const int key0 = 128 * j + 64 * hf;
          if (key0 + 63 > lim) {   // causal mask (and padding rows: every key)
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (key0 + c > lim) x[c] = -INFINITY;
          }
          float mq[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
          for (int c = 4; c < 64; c += 4) {
            mq[0] = fmaxf(mq[0], x[c]);
            mq[1] = fmaxf(mq[1], x[c + 1]);
            mq[2] = fmaxf(mq[2], x[c + 2]);
            mq[3] = fmaxf(mq[3], x[c + 3]);
          }
          const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
          const float m_cand = fmaxf(m_run, mt * sl2);
          const bool grow = m_cand > m_run + kPfRescale;   // also the first finite maximum
          float alpha = 1.f;
          if (grow) {
            alpha = (m_run == -INFINITY) ? 0.f : ex2f(m_run - m_cand);
            m_run = m_cand;
          }
          // O_hf holds this half's value sums of tiles < j: rescale the rows
          // whose maximum grew, once the value MMAs of tile j - 1 are complete
          if (__any_sync(0xffffffffu, grow && l_run > 0.f)) {
            ok = warp_ok(mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_flag, kPfWaitNs),
                         abort_flag, a.err);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float o[32];
              const uint32_t oc = tmem + lane_off + kTO + hf * 128 + 32 * c;
              tmem_ld32(oc, o);
              tmem_ld_wait();
              uint32_t u[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(o[e] * alpha);
              tmem_st32(oc, u);
            }
            tmem_st_wait();
          }
          l_run *= alpha;
          const float mu = (m_run == -INFINITY) ? 0.f : m_run;
          // probabilities as bf16 pairs over the first 32 columns of this
          // half's scores (already read into registers)
          float sq[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2f(fmaf(x[2 * c], sl2, -mu)), p1 = ex2f(fmaf(x[2 * c + 1], sl2, -mu));
            sq[c & 3] += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
          }
          tmem_st32(sbuf, pk);
          tmem_st_wait();
          l_run += (sq[0] + sq[1]) + (sq[2] + sq[3]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[s]);
        }
        if (!ok) break;
        const uint32_t g_last = g0 + n_kt - 1;
        g0 += n_kt;
        ++nq;
        // the next item: its query tile is rotated now, so that its first
        // score MMAs run while this item's outputs are written
        ++n;
        int nxt;
        ok = warp_ok(fetch(n, &nxt), abort_flag, a.err);
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[n & 1]);
        AtItem it2{};
        int n_kt2 = 0;
        if (nxt >= 0) {
          it2 = at_item(nxt, n_qt, a.H);
          n_kt2 = at_key_tiles(a, it2);
          if (n_kt2 > 0 && !rotate(it2, nq)) {
            ok = false;
            break;
          }
        }
        // epilogue: merge the two halves, o = (O_0 a_0 + O_1 a_1) / (l_0 a_0 + l_1 a_1)
        // with a_h = 2^(m_h - m), lse = (m + log2 l) ln 2.  Half hf writes
        // output columns 64 hf .. 64 hf + 63.
        ok = warp_ok(mbar_wait(&pv_done[g_last & 1], (g_last >> 1) & 1, abort_flag, kPfWaitNs), abort_flag,
                     a.err);
        if (!ok) break;
        row_m[hf][r] = m_run;
        row_l[hf][r] = l_run;
        __syncwarp();
        if (lane == 0) mbar_arrive(&grp);
        ok = warp_ok(mbar_wait(&grp, (nq - 1) & 1, abort_flag, kPfWaitNs), abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        const float m0 = row_m[0][r], m1 = row_m[1][r];
        float m = fmaxf(m0, m1);
        if (m == -INFINITY) m = 0.f;   // padding rows
        const float a0 = ex2f(m0 - m), a1 = ex2f(m1 - m);
        const float l = row_l[0][r] * a0 + row_l[1][r] * a1;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float f0 = a0 * inv, f1 = a1 * inv;
        const int row0 = it.qt * 128 + 32 * q4;   // first query of this warp's rows
        float* obase = a.o + (((size_t)it.b * a.T_q + row0) * a.H + it.h) * a.d_h + 64 * hf;
        const size_t ostride = (size_t)a.H * a.d_h;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float o0[32], o1[32];
          tmem_ld32(tmem + lane_off + kTO + 64 * hf + 32 * c, o0);
          tmem_ld32(tmem + lane_off + kTO + 128 + 64 * hf + 32 * c, o1);
          tmem_ld_wait();
          if (c == 1) {   // both halves' outputs read: the next item's value MMAs may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free);
          }
          // 8 columns at a time through this warp's buffer, so that each
          // store instruction writes 16 rows x 32 contiguous bytes (one row
          // per thread would write 32 rows x 16 bytes): row i's two 16-byte
          // halves sit at i * 32 + 16 (k ^ ((i >> 2) & 1)), conflict-free both ways
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int e = 8 * q + 4 * k;
              *reinterpret_cast<float4*>(ebuf + lane * 32 + ((k ^ ((lane >> 2) & 1)) << 4)) =
                  make_float4(o0[e] * f0 + o1[e] * f1, o0[e + 1] * f0 + o1[e + 1] * f1,
                              o0[e + 2] * f0 + o1[e + 2] * f1, o0[e + 3] * f0 + o1[e + 3] * f1);
            }
            __syncwarp();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int i = 16 * h2 + (lane >> 1), k = lane & 1;
              const float4 v = *reinterpret_cast<const float4*>(ebuf + i * 32 + ((k ^ ((i >> 2) & 1)) << 4));
              if (row0 + i < a.T_q) *reinterpret_cast<float4*>(obase + i * ostride + 32 * c + 8 * q + 4 * k) = v;
            }
            __syncwarp();
          }
        }
        if (hf == 0 && t < a.T_q && a.lse) a.lse[qrow * a.H + it.h] = (m + log2f(l)) * kPfLn2;
        cur = nxt;
        it = it2;
        n_kt = n_kt2;
        continue;
      }
      // an item without key tiles: on to the next
      ++n;
      ok = warp_ok(fetch(n, &cur), abort_flag, a.err);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[n & 1]);
      if (cur >= 0) {
        it = at_item(cur, n_qt, a.H);
        n_kt = at_key_tiles(a, it);
        if (n_kt > 0) ok = rotate(it, nq);
      }
    }
  }

  // ---- drain: MMAs complete, copies landed, then free TMEM
  __syncwarp();
  if (warp == 1 && lane == 0) {
    mma_commit(&mma_final);
    if (!mbar_wait(&mma_final, 0, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
  }
  if (warp == 0 && lane == 0) {
    if (n_q > 0 && !mbar_wait(&q_full, (n_q - 1) & 1, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
    for (uint32_t k = 0; k < (uint32_t)kAtStages && k < n_k; ++k) {
      const uint32_t j = n_k - 1 - k;
      if (!mbar_wait(&k_full[j & 1], (j >> 1) & 1, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
    }
    for (uint32_t k = 0; k < (uint32_t)kAtStages && k < n_v; ++k) {
      const uint32_t j = n_v - 1 - k;
      if (!mbar_wait(&v_full[j & 1], (j >> 1) & 1, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && slot >= 0) {
    // every CTA has taken its last item: the last one out zeroes the counters
    __threadfence();
    if (atomicAdd(&g_at_work[slot][1], 1u) == gridDim.x - 1) {
      g_at_work[slot][0] = 0;
      g_at_work[slot][1] = 0;
      __threadfence();
    }
  }
}

}  // namespace

bool prefill_supported(int dtype, int d_c, int d_r, int d_h) {
  return dtype == BF16 && d_c == 512 && d_r == 64 && d_h == 128;
}

int prefill_kv_rows(int max_blocks) {
  const long long rows = (long long)max_blocks * kPage;
  return (int)((rows + 127) / 128 * 128);
}

cudaError_t launch_prefill_kv(const PrefillKvArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  TensorMapEncodeFn enc = nullptr;
  cudaError_t e = tensor_map_encoder(&enc);
  if (e != cudaSuccess) return e;
  const int D = a.d_c + a.d_r;
  CUtensorMap tm_pool, tm_wuk, tm_wuv;
  {
    // the pool [num_blocks * 64 rows, D]: box of 64 columns x 64 rows (one page)
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)a.num_blocks * kPage};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tm_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.cache), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const void* ws[2] = {a.w_uk, a.w_uv};
  CUtensorMap* tms[2] = {&tm_wuk, &tm_wuv};
  for (int i = 0; i < 2; ++i) {
    // W [H * d_h, d_c]: box of 64 columns x 128 rows (one head)
    cuuint64_t dims[2] = {(cuuint64_t)a.d_c, (cuuint64_t)a.H * a.d_h};
    cuuint64_t strides[1] = {(cuuint64_t)a.d_c * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    if (enc(tms[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ws[i]), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  e = cudaFuncSetAttribute(prefill_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.R / 128, a.B, (a.H + kKvHeads - 1) / kKvHeads);
  prefill_kv_kernel<<<grid, kPfThreads, kKvSmem, s>>>(a, tm_pool, tm_wuk, tm_wuv);
  return cudaGetLastError();
}

namespace {

// SM count of the current device (cached per device)
cudaError_t device_sm_count(int* sms) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *sms = c;
      return cudaSuccess;
    }
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev].store(*sms, std::memory_order_relaxed);
  return e;
}

// The attention kernel's CTAs take work items from a counter in device
// memory.  Launches on one stream run one after another, so each stream (of
// each device) gets a counter of its own; the kernel leaves it at zero.  Past
// kAtSlots streams, or on the per-thread default stream (one handle shared by
// concurrently running host threads), the CTAs take items in a fixed order
// instead (-1).
int work_slot(cudaStream_t s) {
  if (s == cudaStreamPerThread) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  static std::mutex mu;
  static cudaStream_t owner[64][kAtSlots];
  static int used[64];
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used[dev]; ++i)
    if (owner[dev][i] == s) return i;
  if (used[dev] == kAtSlots) return -1;
  owner[dev][used[dev]] = s;
  return used[dev]++;
}

}  // namespace

cudaError_t launch_prefill_attn(const PrefillAttnArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  TensorMapEncodeFn enc = nullptr;
  cudaError_t e = tensor_map_encoder(&enc);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_q, tm_k, tm_kr, tm_v;
  const auto map3 = [&](CUtensorMap* tm, const void* base, long long rows) -> bool {
    // q_nope [B * T_q, H, 128] as a 3-D tensor: box of 64 dims x 1 head x 128 rows
    cuuint64_t dims[3] = {(cuuint64_t)a.d_h, (cuuint64_t)a.H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)a.d_h * 2, (cuuint64_t)a.H * a.d_h * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const long long kv_rows = (long long)a.B * a.R;
  if (!map3(&tm_q, a.q_nope, (long long)a.B * a.T_q)) return cudaErrorInvalidValue;
  CUtensorMap tm_qr;
  {
    // q_rope [B * T_q, H, 64] unrotated: box of 64 dims x 1 head x 128 rows
    cuuint64_t dims[3] = {(cuuint64_t)a.d_r, (cuuint64_t)a.H, (cuuint64_t)a.B * a.T_q};
    cuuint64_t strides[2] = {(cuuint64_t)a.d_r * 2, (cuuint64_t)a.H * a.d_r * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_qr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q_rope), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }

  const void* kvs[2] = {a.k_nope, a.v};
  CUtensorMap* kvm[2] = {&tm_k, &tm_v};
  for (int i = 0; i < 2; ++i) {
    // k_nope, v [B, H, R, d_h = 128] as 3-D (64 dims, B * H * R rows, 2 halves
    // of d_h): one box of 64 dims x 128 rows x 2 halves is a whole key tile of
    // a head (32 KB) in ONE copy, laid out [half][row][64 dims] as the MMA
    // reads it (every copy instruction costs the SM's copy engine ~0.3 us, so
    // the tile is not split into two boxes)
    cuuint64_t dims[3] = {64, (cuuint64_t)kv_rows * a.H, (cuuint64_t)a.d_h / 64};
    cuuint64_t strides[2] = {(cuuint64_t)a.d_h * 2, 128};
    cuuint32_t box[3] = {64, 128, 2};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(kvm[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kvs[i]), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // k_rope [rows, 64]: box of 64 dims x 128 rows
    cuuint64_t dims[2] = {(cuuint64_t)a.d_r, (cuuint64_t)kv_rows};
    cuuint64_t strides[1] = {(cuuint64_t)a.d_r * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tm_kr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.k_rope), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const RopeFreqs fr = rope_freqs(a.rope_base, a.d_r);
  e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAtSmem);
  if (e != cudaSuccess) return e;
  // one CTA per SM (the rings fill shared memory), each taking work items
  // until none are left
  const long long n_items = (long long)((a.T_q + 127) / 128) * a.H * a.B;
  if (n_items > INT32_MAX) return cudaErrorInvalidValue;
  int sms = 0;
  e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<long long>(n_items, sms);
  prefill_attn_kernel<<<grid, kAtThreads, kAtSmem, s>>>(a, tm_q, tm_qr, tm_k, tm_kr, tm_v, fr,
                                                        work_slot(s), (int)n_items);
  return cudaGetLastError();
}

}  // namespace mla
