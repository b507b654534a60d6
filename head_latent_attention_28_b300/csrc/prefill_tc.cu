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
//    128 x 512); the row warps copy them into TMEM, where they stay as the
//    MMA's A operand for all heads of the group, and the shared memory they
//    used becomes output staging.  W^UK_h and W^UV_h (128 x 512 each) stream
//    in 64-column chunks through a six-unit ring; tcgen05.mma with M = 128
//    rows, N = 128, K = 512 accumulates k_h and then v_h in two TMEM
//    accumulators, so the epilogue of one overlaps the MMAs of the other.
//    Four warps convert to bf16 and write k_nope[b, h, s, :] and
//    v[b, h, s, :] through the staging area, 512 contiguous bytes per store
//    instruction; rows past the sequence end inside its last tile are written
//    as zeros.  The first head
//    group also copies the rotated rotary key R_s k^R_s of each row.  For a
//    chunk of a chunked prefill only the chunk's rows [L - T_new, L) are
//    written (tiles below them exit at once); earlier rows stay as the
//    earlier chunks wrote them.
//  * prefill_attn_kernel: persistent, one CTA per SM, each taking work items
//    (query tiles 2p and 2p + 1 of one head of one sequence; the items of a
//    head one after another, latest pair first) from a counter until none
//    are left.  Both query tiles of an item share every key and value tile,
//    so each tile brought into shared memory feeds twice the MMA work of one
//    query tile.  Scores over d_h + d^R_h = 192 dims (M = 128 queries,
//    N = 128 keys) of query tile x go into TMEM columns 128 x; four softmax
//    warps per query tile (thread = query row) run a base-2 online softmax
//    with a lazy running max (the output is rescaled only when a row maximum
//    grows by more than 2^8; exact after the final division), write bf16
//    probabilities over the second half of their scores and accumulate
//    O_x += P_x V in TMEM (P read from TMEM as the tcgen05.mma A operand).
//    The MMA issuer interleaves the two query tiles (S_0(j+1) runs while
//    tile 1's softmax of key tile j does).  Key tiles stream through a
//    two-stage ring and value tiles through one buffer, each with a producer
//    warp of its own; both run on from one item into the next.  The query's
//    rotary half is copied unrotated and rotated in place (the same
//    fixed-point angle table as the query absorption).  Outputs leave through
//    the value buffer once an item's MMAs are done, so that each store
//    instruction writes 4 rows x 128 contiguous bytes.
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
constexpr int kKvA = 8 * kBox16;         // 128 rows x 512 latents (then the output staging)
constexpr int kKvUnits = 6;              // weight ring: 64-column chunks of W^UK_h or W^UV_h
constexpr int kKvW = kBox16;             // one chunk: 128 rows x 64 latents
constexpr int kKvE = 8192;               // per row warp: 32 rows x 256 bytes of output staging
constexpr int kKvSmem = kKvA + kKvUnits * kKvW + 1024;
// TMEM columns: the K and V accumulators of the current head, then the
// latent tile as the MMA A operand (a row per lane, bf16 pairs per column)
constexpr uint32_t kKvAccK = 0, kKvAccV = 128, kKvTA = 256;

__global__ void __launch_bounds__(kPfThreads, 1)
prefill_kv_kernel(const PrefillKvArgs a, const __grid_constant__ CUtensorMap tm_pool,
                  const __grid_constant__ CUtensorMap tm_wuk, const __grid_constant__ CUtensorMap tm_wuv) {
  extern __shared__ uint8_t kv_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(kv_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t a_full, a_ready, w_full[kKvUnits], w_empty[kKvUnits], d_full[2], d_empty[2], mma_final;
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
    mbar_init(&a_ready, 4);
    for (int u = 0; u < kKvUnits; ++u) {
      mbar_init(&w_full[u], 1);
      mbar_init(&w_empty[u], 1);
    }
    for (int d = 0; d < 2; ++d) {   // d = 0: the K accumulator, 1: the V accumulator
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
      // per head: the 8 chunks of W^UK_h, then the 8 of W^UV_h
      for (int hh = 0; hh < nh; ++hh) {
        const int wrow = (h0 + hh) * a.d_h;
        for (int part = 0; part < 2; ++part) {
          for (int c = 0; c < 8; ++c) {
            const uint32_t g = n_issued, u = g % kKvUnits;
            if (g >= (uint32_t)kKvUnits &&
                !mbar_wait(&w_empty[u], ((g / kKvUnits) - 1) & 1, abort_flag, kPfWaitNs)) {
              *abort_flag = 1;
              atomicOr(a.err, kErrTimeout);
              break;
            }
            mbar_arrive_expect_tx(&w_full[u], kKvW);
            tma_load_2d(sW + u * kKvW, part == 0 ? &tm_wuk : &tm_wuv, &w_full[u], 64 * c, wrow, pol_w);
            ++n_issued;
          }
          if (*abort_flag) break;
        }
        if (*abort_flag) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // k_h = W^UK_h c and v_h = W^UV_h c as two M = 128, N = 128, K = 512
      // products with the latent tile read from TMEM: the epilogue of one
      // part overlaps the MMAs of the other
      const uint32_t id = idesc_bf16_f32(128, 128, 0, 0);   // A from TMEM, B K-major
      bool ok = mbar_wait(&a_ready, 0, abort_flag, kPfWaitNs);
      uint32_t g = 0;
      for (int hh = 0; ok && hh < nh; ++hh) {
        for (int part = 0; ok && part < 2; ++part) {
          if (hh >= 1) ok = mbar_wait(&d_empty[part], (hh - 1) & 1, abort_flag, kPfWaitNs);
          for (int c = 0; ok && c < 8; ++c, ++g) {
            const uint32_t u = g % kKvUnits;
            ok = mbar_wait(&w_full[u], (g / kKvUnits) & 1, abort_flag, kPfWaitNs);
            if (!ok) break;
            tc_fence_after();
            const uint8_t* wb = sW + u * kKvW;
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // latents 64 c + 16 q .. + 15
              const uint64_t bd = sdesc_sw128(smem_u32(wb + q * 32), 16, 1024);
              mma_ts(tmem + (part ? kKvAccV : kKvAccK), tmem + kKvTA + 32 * c + 8 * q, bd, id,
                     (c > 0 || q > 0) ? 1 : 0);
            }
            mma_commit(&w_empty[u]);
          }
          if (ok) mma_commit(&d_full[part]);
        }
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
    bool ok = warp_ok(mbar_wait(&a_full, 0, abort_flag, kPfWaitNs), abort_flag, a.err);
    if (ok) {
      // the latent row into TMEM columns kKvTA.. (bf16 pairs): chunk c of the
      // tile (64 latents, 128-byte swizzled rows) into columns 32 c .. 32 c + 31
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t w[32];
        const uint8_t* src = sA + c * kBox16 + r * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + ((k ^ (r & 7)) << 4));
          w[4 * k] = v.x;
          w[4 * k + 1] = v.y;
          w[4 * k + 2] = v.z;
          w[4 * k + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + kKvTA + 32 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_ready);
    }
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
    // a head's 32 rows of k_nope (then of v) are 8 KB of contiguous memory:
    // they go out through this warp's staging rows in the (now free) latent
    // buffer (row i's 16-byte chunk k at i * 256 + 16 (k ^ (i & 15)),
    // conflict-free both ways), so that each store instruction writes 512
    // contiguous bytes (one row per thread would write 32 rows x 16 bytes)
    uint8_t* stage = sA + q4 * kKvE;
    const int wrow0 = r0 + 32 * q4;   // this warp's first row
    for (int hh = 0; ok && hh < nh; ++hh) {
      const size_t off = (((size_t)b * a.H + (h0 + hh)) * a.R + wrow0) * a.d_h;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {   // k_nope, then v
        ok = warp_ok(mbar_wait(&d_full[part], hh & 1, abort_flag, kPfWaitNs), abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          float x[32];
          tmem_ld32(tmem + lane_off + (part ? kKvAccV : kKvAccK) + 32 * c4, x);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (real)
              w = make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]), pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                             pack_bf16x2(x[8 * i + 4], x[8 * i + 5]), pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
            const int k = 4 * c4 + i;
            *reinterpret_cast<uint4*>(stage + lane * 256 + ((k ^ (lane & 15)) << 4)) = w;
          }
        }
        // the accumulator is read: the next head's MMAs of this part may reuse it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[part]);
        uint8_t* gbase = reinterpret_cast<uint8_t*>(part == 0 ? a.k_nope : a.v) + off * 2;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int rr = 2 * i + (lane >> 4), k = lane & 15;
          const uint4 w = *reinterpret_cast<const uint4*>(stage + rr * 256 + ((k ^ (rr & 15)) << 4));
          if (wrow0 + rr >= row_lo) *reinterpret_cast<uint4*>(gbase + rr * 256 + k * 16) = w;
        }
        __syncwarp();
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
    if (!mbar_wait(&a_full, 0, never, kPfWaitNs)) atomicOr(a.err, kErrTimeout);
    for (uint32_t k = 0; k < (uint32_t)kKvUnits && k < n_issued; ++k) {
      const uint32_t g = n_issued - 1 - k;
      if (!mbar_wait(&w_full[g % kKvUnits], (g / kKvUnits) & 1, never, kPfWaitNs))
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
constexpr int kAtV = 2 * kBox16;         // value tile (its buffer also stages the outputs)
constexpr int kAtStages = 2;             // key ring
constexpr int kAtOffK = 2 * kAtQ;
constexpr int kAtOffV = kAtOffK + kAtStages * kAtK;
constexpr int kAtSmem = kAtOffV + kAtV + 1024;
constexpr int kAtThreads = 352;          // 11 warps: key producer, MMA issuer, 2 x 4 row warps, value producer
// TMEM columns: the scores of query tile X at 128 X (its probabilities
// overwrite the last 64 columns), its output accumulator at 256 + 128 X
constexpr uint32_t kTS = 0, kTO = 256;
constexpr int kAtSlots = 64;             // work counters: one per stream that launches the kernel

// work counters of the persistent attention kernel: [0] next item, [1] CTAs
// finished (the last CTA to finish zeroes both for the next launch)
__device__ unsigned g_at_work[kAtSlots][2];

// a work item: query tiles 2p and 2p + 1 (the second may not exist) of one
// head of one sequence.  Items are numbered head by head (so the CTAs running
// at any time share the keys and values of a few heads in L2), latest pair
// first within a head (it sees the most keys).
struct AtItem {
  int p, h, b;
};
__device__ __forceinline__ AtItem at_item(int i, int n_pairs, int H) {
  const int hb = i / n_pairs;
  return AtItem{n_pairs - 1 - (i - hb * n_pairs), hb % H, hb / H};
}
// key tiles query tile qt sees (0 past the last tile, or for a sequence of
// invalid length): keys 0 .. position of the tile's last query
__device__ __forceinline__ int at_key_tiles(const PrefillAttnArgs& a, int b, int qt) {
  const int L = a.seqlens[b];
  if (qt * 128 >= a.T_q || L < a.T_q || L > a.max_len) return 0;
  const int last_t = min(qt * 128 + 127, a.T_q - 1);
  return (L - a.T_q + last_t) / 128 + 1;
}

// Persistent: each CTA takes work items (from a counter when `slot` >= 0, else
// items blockIdx.x, blockIdx.x + gridDim.x, ...) until none are left.  The key
// producer publishes each item to the other roles through a two-entry ring.
// An item's two query tiles share every key and value tile (half the bytes
// per score of one tile per CTA).  The MMA issuer runs S_0(0) S_1(0), then per
// key tile j PV_0(j) S_0(j+1) PV_1(j) S_1(j+1), so that one query tile's
// scores run while the other's softmax does.  Key tiles stream through a
// two-stage ring and value tiles through one buffer (shared memory holds no
// more beside two query tiles), each with a producer warp of its own; both run
// on from one item into the next.  The next item's query tiles load as soon as
// the last score MMA of the current one has read the old ones; the row warps
// rotate them between their last softmax and their output stores, so the next
// item's first score MMAs overlap those stores.  The outputs leave through the
// value buffer (free once the item's last value MMAs are done, refilled once
// every row warp is done with it), so that each store instruction writes
// 4 rows x 128 bytes.
__global__ void __launch_bounds__(kAtThreads, 1)
prefill_attn_kernel(const PrefillAttnArgs a, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ RopeFreqs fr, int slot, int n_items) {
  extern __shared__ uint8_t at_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t q_full, q_ready[2], q_free, k_full[kAtStages], k_empty[kAtStages], v_full, v_empty,
      s_full[2], p_full[2], pv_done[2], o_free[2], item_done, epi_done, mma_final, item_full[2], item_empty[2];
  __shared__ int item_id[2];
  __shared__ uint32_t tbase;
  __shared__ int abort_raw, never_raw;
  volatile int* abort_flag = &abort_raw;
  volatile int* never = &never_raw;
  volatile int* items = item_id;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (a.T_q + 127) / 128;
  const int n_pairs = (n_qt + 1) / 2;

  if (threadIdx.x == 0) {
    abort_raw = 0;
    never_raw = 0;
    mbar_init(&q_full, 1);
    mbar_init(&q_free, 1);
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    mbar_init(&v_full, 1);
    mbar_init(&v_empty, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_ready[x], 4);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&pv_done[x], 1);
      mbar_init(&o_free[x], 4);
      mbar_init(&item_full[x], 1);
      mbar_init(&item_empty[x], 10);   // the MMA issuer, the 8 row warps and the value producer
    }
    mbar_init(&item_done, 1);
    mbar_init(&epi_done, 8);
    mbar_init(&mma_final, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 1) tmem_alloc(&tbase, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  uint8_t* sK = smem + kAtOffK;
  uint8_t* sV = smem + kAtOffV;
  uint32_t n_k = 0, n_v = 0, n_q = 0;          // producers: key, value and query loads issued

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
        const AtItem it = at_item(i, n_pairs, a.H);
        const int nk0 = at_key_tiles(a, it.b, 2 * it.p), nk1 = at_key_tiles(a, it.b, 2 * it.p + 1);
        const int n_kt = max(nk0, nk1);
        const int krow0 = (it.b * a.H + it.h) * a.R;   // first row of (sequence, head) in k_nope and v
        const int rrow0 = it.b * a.R;                  // first row of the sequence in k_rope
        const int tok0 = it.b * a.T_q + 256 * it.p;    // the first query tile's first row in q_nope
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
            // the query tiles, once the last score MMA of the previous item has read the old ones
            ok = n_q == 0 || mbar_wait(&q_free, (n_q - 1) & 1, abort_flag, kPfWaitNs);
            if (!ok) break;
            const int nt = nk1 > 0 ? 2 : 1;
            mbar_arrive_expect_tx(&q_full, nt * kAtQ);
            for (int x = 0; x < nt; ++x) {
              uint8_t* qd = smem + x * kAtQ;
              tma_load_3d(qd, &tm_q, &q_full, 0, it.h, tok0 + 128 * x, pol_q);
              tma_load_3d(qd + kBox16, &tm_q, &q_full, 64, it.h, tok0 + 128 * x, pol_q);
              tma_load_3d(qd + 2 * kBox16, &tm_qr, &q_full, 0, it.h, tok0 + 128 * x, pol_q);   // rotated in place
            }
            ++n_q;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMAs issued by one thread run in issue order: the scores of query
      // tile x for key tile j + 1 overwrite its probabilities of tile j only
      // after the value MMAs of tile j (issued earlier) have read them
      const uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);   // Q, K both K-major
      const uint32_t idO = idesc_bf16_f32(128, 128, 0, 1);   // P from TMEM, V MN-major
      bool ok = true;
      uint32_t g = 0, nq = 0;                  // key tiles and items with key tiles consumed
      uint32_t cnt0 = 0, cnt1 = 0;             // key tiles each query tile has consumed
      for (uint32_t n = 0; ok; ++n) {
        int i;
        ok = fetch(n, &i);
        if (!ok) break;
        mbar_arrive(&item_empty[n & 1]);
        if (i < 0) break;
        const AtItem it = at_item(i, n_pairs, a.H);
        const int nk0 = at_key_tiles(a, it.b, 2 * it.p), nk1 = at_key_tiles(a, it.b, 2 * it.p + 1);
        const int n_kt = max(nk0, nk1);
        if (n_kt == 0) continue;
        ok = mbar_wait(&q_full, nq & 1, abort_flag, kPfWaitNs);
        // key tile j is seen by query tile x when j < nk_x (nk1 >= nk0 unless
        // the second tile does not exist)
        const auto sees = [&](int x, int j) { return j < (x ? nk1 : nk0); };
        // S_x(j): scores of query tile x against key tile j; the first score
        // MMA of a key tile waits for it, the last frees its slot
        const auto score = [&](int x, int j) -> bool {
          const uint32_t gj = g + j, s = gj & 1;
          if ((x == 0 || !sees(0, j)) && !mbar_wait(&k_full[s], (gj >> 1) & 1, abort_flag, kPfWaitNs)) return false;
          if (j == 0 && !mbar_wait(&q_ready[x], nq & 1, abort_flag, kPfWaitNs)) return false;
          tc_fence_after();
          const uint8_t* qd = smem + x * kAtQ;
          const uint8_t* kd = sK + s * kAtK;
#pragma unroll
          for (int kk = 0; kk < 12; ++kk) {
            const uint64_t ad = sdesc_sw128(smem_u32(qd + (kk >> 2) * kBox16 + (kk & 3) * 32), 16, 1024);
            const uint64_t bd = sdesc_sw128(smem_u32(kd + (kk >> 2) * kBox16 + (kk & 3) * 32), 16, 1024);
            mma_ss(tmem + kTS + 128 * x, ad, bd, idS, kk > 0 ? 1 : 0);
          }
          mma_commit(&s_full[x]);
          if (x == 1 || !sees(1, j)) {
            mma_commit(&k_empty[s]);
            if (j == n_kt - 1) mma_commit(&q_free);
          }
          return true;
        };
        // O_x += P_x(j) V(j); the first value MMA of a tile waits for it, the
        // last frees the value buffer
        const auto value = [&](int x, int j) -> bool {
          const uint32_t gj = g + j;
          if ((x == 0 || !sees(0, j)) && !mbar_wait(&v_full, gj & 1, abort_flag, kPfWaitNs)) return false;
          if (!mbar_wait(&p_full[x], ((x ? cnt1 : cnt0) + j) & 1, abort_flag, kPfWaitNs)) return false;
          // the first value MMAs of an item overwrite the output: the row
          // warps must have read the previous item's
          if (j == 0 && nq > 0 && !mbar_wait(&o_free[x], (nq - 1) & 1, abort_flag, kPfWaitNs)) return false;
          tc_fence_after();
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {   // 16 keys per step
            const uint64_t bd = sdesc_sw128(smem_u32(sV + k8 * 2048), kBox16, 1024);
            mma_ts(tmem + kTO + 128 * x, tmem + kTS + 128 * x + 64 + 8 * k8, bd, idO, (j > 0 || k8 > 0) ? 1 : 0);
          }
          mma_commit(&pv_done[x]);
          if (x == 1 || !sees(1, j)) mma_commit(&v_empty);
          return true;
        };
        // issue order S_0(0) S_1(0), then per key tile j: PV_0(j) S_0(j+1)
        // PV_1(j) S_1(j+1), so that each query tile's scores for the next key
        // tile run while the other tile's softmax does
        for (int x = 0; ok && x < 2; ++x)
          if (sees(x, 0)) ok = score(x, 0);
        for (int j = 0; ok && j < n_kt; ++j) {
          for (int x = 0; ok && x < 2; ++x) {
            if (sees(x, j)) ok = value(x, j);
            if (ok && sees(x, j + 1)) ok = score(x, j + 1);
          }
        }
        g += n_kt;
        if (!ok) break;
        mma_commit(&item_done);
        cnt0 += nk0;
        cnt1 += nk1;
        ++nq;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else if (warp == kAtThreads / 32 - 1) {
    // value tiles have a producer of their own: the single value buffer is
    // refilled only once both query tiles' value MMAs have read it, and the
    // key tiles must not wait behind that
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();
      bool ok = true;
      uint32_t nq = 0;                         // items with key tiles
      for (uint32_t n = 0; ok; ++n) {
        int i;
        ok = fetch(n, &i);
        if (!ok) break;
        mbar_arrive(&item_empty[n & 1]);
        if (i < 0) break;
        const AtItem it = at_item(i, n_pairs, a.H);
        const int n_kt = max(at_key_tiles(a, it.b, 2 * it.p), at_key_tiles(a, it.b, 2 * it.p + 1));
        const int krow0 = (it.b * a.H + it.h) * a.R;
        for (int j = 0; ok && j < n_kt; ++j) {
          // free once the value MMAs of the previous tile are done and, for an
          // item's first tile, once every row warp has stored the previous
          // item's outputs through it
          ok = n_v == 0 || mbar_wait(&v_empty, (n_v - 1) & 1, abort_flag, kPfWaitNs);
          if (ok && j == 0 && nq > 0) ok = mbar_wait(&epi_done, (nq - 1) & 1, abort_flag, kPfWaitNs);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full, kAtV);
          tma_load_3d(sV, &tm_v, &v_full, 0, krow0 + 128 * j, 0, pol_kv);
          ++n_v;
        }
        if (n_kt > 0) ++nq;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else {
    // row warps: query tile x (warps 2-5: the item's first tile, 6-9: its
    // second) runs a base-2 online softmax over all 128 keys of every key
    // tile into its output accumulator O_x; thread = query row r (TMEM lane r)
    const int x = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float sl2 = a.scale * kPfLog2e;
    uint8_t* qx = smem + x * kAtQ;
    uint8_t* ebuf = sV + (4 * x + q4) * 4096;   // this warp's 32 rows x 128 bytes while storing
    uint32_t cnt = 0, nq = 0;                  // key tiles and items with key tiles consumed
    bool ok = true;

    // the query's rotary half was copied unrotated into box 2 of the query
    // tile (K-major, 128-byte swizzle: 16-byte chunk c of row r sits at chunk
    // c ^ (r & 7)); rotate it in place by the query's position; rows past the
    // sequence become zeros.  A tile that does not exist only signals.
    const auto prologue = [&](const AtItem& it, int nkx, uint32_t q_index) -> bool {
      if (nkx > 0) {
        if (!warp_ok(mbar_wait(&q_full, q_index & 1, abort_flag, kPfWaitNs), abort_flag, a.err)) return false;
        const int t = (2 * it.p + x) * 128 + r;
        const int L = a.seqlens[it.b];
        const bool real = t < a.T_q;
        const uint64_t pos = (uint64_t)(int64_t)(L - a.T_q + t);
        uint8_t* qrow_s = qx + 2 * kBox16 + r * 128;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {   // 16-byte chunk c: rotary pairs 4c .. 4c + 3
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
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_ready[x]);
      return true;
    };
    const auto tiles_of = [&](const AtItem& it, int* nkx) -> int {
      const int n0 = at_key_tiles(a, it.b, 2 * it.p), n1 = at_key_tiles(a, it.b, 2 * it.p + 1);
      *nkx = x == 0 ? n0 : n1;
      return max(n0, n1);
    };

    uint32_t n = 0;
    int cur;
    ok = warp_ok(fetch(n, &cur), abort_flag, a.err);
    if (ok) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[n & 1]);
    }
    AtItem it{};
    int n_kt = 0, nkx = 0;
    if (ok && cur >= 0) {
      it = at_item(cur, n_pairs, a.H);
      n_kt = tiles_of(it, &nkx);
      if (n_kt > 0) ok = prologue(it, nkx, nq);
    }
    while (ok && cur >= 0) {
      const int qt = 2 * it.p + x;
      const int t = qt * 128 + r;
      const int L = a.seqlens[it.b];
      const size_t qrow = (size_t)it.b * a.T_q + t;
      if (n_kt == 0) {
        // a sequence of invalid length: zeros (the error word says why)
        if (it.p == 0 && it.h == 0 && lane == 0 && x == 0 && q4 == 0) atomicOr(a.err, kErrBadIndex);
        if (t < a.T_q) {
          float* orow = a.o + (qrow * a.H + it.h) * a.d_h;
          for (int c = 0; c < 32; ++c) reinterpret_cast<float4*>(orow)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (a.lse) a.lse[qrow * a.H + it.h] = 0.f;
        }
        ++n;
        ok = warp_ok(fetch(n, &cur), abort_flag, a.err);
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[n & 1]);
        if (cur >= 0) {
          it = at_item(cur, n_pairs, a.H);
          n_kt = tiles_of(it, &nkx);
          if (n_kt > 0) ok = prologue(it, nkx, nq);
        }
        continue;
      }
      const int lim = t < a.T_q ? L - a.T_q + t : -1;   // position of the query = its last visible key
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; ok && j < nkx; ++j) {
        const uint32_t g = cnt + j;
        ok = warp_ok(mbar_wait(&s_full[x], g & 1, abort_flag, kPfWaitNs), abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sbuf = tmem + lane_off + kTS + 128 * x;
        const int key0 = 128 * j;
        const bool masked = key0 + 127 > lim;   // causal mask (and padding rows: every key)
        // the row maximum over both 64-key halves, keeping the second half;
        // the first is read again for its probabilities (two halves in
        // registers at once would not fit beside the rest)
        float xb[64];
        float mq[4];
        {
          float xa[64];
          tmem_ld64(sbuf, xa);
          tmem_ld_wait();
          if (masked) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (key0 + c > lim) xa[c] = -INFINITY;
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) mq[c] = xa[c];
#pragma unroll
          for (int c = 4; c < 64; c += 4) {
            mq[0] = fmaxf(mq[0], xa[c]);
            mq[1] = fmaxf(mq[1], xa[c + 1]);
            mq[2] = fmaxf(mq[2], xa[c + 2]);
            mq[3] = fmaxf(mq[3], xa[c + 3]);
          }
        }
        tmem_ld64(sbuf + 64, xb);
        tmem_ld_wait();
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (key0 + 64 + c > lim) xb[c] = -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          mq[0] = fmaxf(mq[0], xb[c]);
          mq[1] = fmaxf(mq[1], xb[c + 1]);
          mq[2] = fmaxf(mq[2], xb[c + 2]);
          mq[3] = fmaxf(mq[3], xb[c + 3]);
        }
        const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        const float m_cand = fmaxf(m_run, mt * sl2);
        const bool grow = m_cand > m_run + kPfRescale;   // also the first finite maximum
        const bool rescale = __any_sync(0xffffffffu, grow && l_run > 0.f);
        float alpha = 1.f;
        if (grow) {
          alpha = (m_run == -INFINITY) ? 0.f : ex2f(m_run - m_cand);
          m_run = m_cand;
        }
        l_run *= alpha;
        const float mu = (m_run == -INFINITY) ? 0.f : m_run;
        // probabilities as bf16 pairs over score columns 64-127: keys 64-127
        // (from registers) into columns 96-127, then keys 0-63 (read again)
        // into columns 64-95
        float sq[4] = {0.f, 0.f, 0.f, 0.f};
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2f(fmaf(xb[2 * c], sl2, -mu)), p1 = ex2f(fmaf(xb[2 * c + 1], sl2, -mu));
            sq[c & 3] += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
          }
          tmem_st32(sbuf + 96, pk);
        }
        {
          float xa[64];
          tmem_ld64(sbuf, xa);
          tmem_ld_wait();
          if (masked) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (key0 + c > lim) xa[c] = -INFINITY;
          }
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2f(fmaf(xa[2 * c], sl2, -mu)), p1 = ex2f(fmaf(xa[2 * c + 1], sl2, -mu));
            sq[c & 3] += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
          }
          tmem_st32(sbuf + 64, pk);
        }
        l_run += (sq[0] + sq[1]) + (sq[2] + sq[3]);
        // O_x holds the value sums of tiles < j: rescale the rows whose
        // maximum grew, once the value MMAs of tile j - 1 are complete (the
        // value MMAs of tile j wait for this warp's signal below)
        if (rescale) {
          ok = warp_ok(mbar_wait(&pv_done[x], (g - 1) & 1, abort_flag, kPfWaitNs), abort_flag, a.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[32];
            const uint32_t oc = tmem + lane_off + kTO + 128 * x + 32 * c;
            tmem_ld32(oc, o);
            tmem_ld_wait();
            uint32_t u[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(o[e] * alpha);
            tmem_st32(oc, u);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
      }
      if (!ok) break;
      cnt += nkx;
      ++nq;
      const AtItem done_it = it;
      const int done_nkx = nkx;
      // the next item: its query tile is rotated now, so that its first
      // score MMAs run while this item's outputs are written
      ++n;
      ok = warp_ok(fetch(n, &cur), abort_flag, a.err);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[n & 1]);
      if (cur >= 0) {
        it = at_item(cur, n_pairs, a.H);
        n_kt = tiles_of(it, &nkx);
        if (n_kt > 0 && !prologue(it, nkx, nq)) {
          ok = false;
          break;
        }
      }
      // epilogue, once every MMA of the item is done (the value buffer is
      // then free): o = O_x / l, lse = (m + log2 l) ln 2
      ok = warp_ok(mbar_wait(&item_done, (nq - 1) & 1, abort_flag, kPfWaitNs), abort_flag, a.err);
      if (!ok) break;
      tc_fence_after();
      if (done_nkx > 0) {
        const float m = m_run == -INFINITY ? 0.f : m_run;   // padding rows
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const int row0 = (2 * done_it.p + x) * 128 + 32 * q4;   // first query of this warp's rows
        float* obase = a.o + (((size_t)done_it.b * a.T_q + row0) * a.H + done_it.h) * a.d_h;
        const size_t ostride = (size_t)a.H * a.d_h;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_off + kTO + 128 * x + 32 * c, o);
          tmem_ld_wait();
          if (c == 3) {   // the outputs are read: the next item's value MMAs may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[x]);
          }
          // 32 columns through this warp's staging rows: row i's 16-byte
          // chunk k sits at i * 128 + 16 (k ^ (i & 7)), conflict-free both
          // ways; each store instruction then writes 4 rows x 128 bytes
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(ebuf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv, o[4 * k + 3] * inv);
          __syncwarp();
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const int i = 4 * i4 + (lane >> 3), k = lane & 7;
            const float4 v = *reinterpret_cast<const float4*>(ebuf + i * 128 + ((k ^ (i & 7)) << 4));
            if (row0 + i < a.T_q) *reinterpret_cast<float4*>(obase + i * ostride + 32 * c + 4 * k) = v;
          }
          __syncwarp();
        }
        if (t < a.T_q && a.lse) a.lse[qrow * a.H + done_it.h] = (m + log2f(l_run)) * kPfLn2;
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free[x]);
      }
      // the value buffer may be refilled
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&epi_done);
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
  }
  if (warp == kAtThreads / 32 - 1 && lane == 0 && n_v > 0 && !mbar_wait(&v_full, (n_v - 1) & 1, never, kPfWaitNs))
    atomicOr(a.err, kErrTimeout);
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
    // a head (32 KB), landing in one copy as [half][row][64 dims], as the MMA
    // reads it
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
  const long long n_items = (long long)((a.T_q + 255) / 256) * a.H * a.B;   // pairs of query tiles
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
