// Tensor-core MLA decode for sm_103a: query rows (heads x query tokens) of a
// sequence in groups of up to 128, cached rows of 512 latent + 64 rotary
// bfloat16 numbers.  The MMAs always run M = 128 rows; fewer rows are zero
// padding, masked out and never written.  A sequence with more than 128 rows
// is split into row groups, each a work item of its own over the same pages.
//
// What it computes is the latent-space attention of the absorbed MLA path
// ("Attention, Part 2: MQA, GQA and MLA", the absorbed inference path: score =
// latent query . latent + rotary query . rotary key, scaled, causal mask,
// softmax, value sum over the latents; "How DeepSeek Rewrote the Transformer":
// the value is the first d_c numbers of the cached row).
//
// How (B300-specific).  One split worker is a cluster of two CTAs on two SMs:
//  * CTA 0, the score CTA, streams its pages from HBM two at a time through a
//    ring of six 16 KB cells (cell c of a page pair = the 64-dim box c of
//    both pages, so one N=128 MMA covers both pages), and computes
//    S = Q . C^T (M=128 rows, N=128 tokens, K=576) with tcgen05.mma into one of
//    two TMEM score buffers.  The latent part of the query (K 0..511) is the A
//    operand in tensor memory, the rotary part (K 512..575) sits in shared
//    memory.  Eight softmax warps (one page of the pair per half) run a
//    base-2 online softmax with a lazy running max (the output is rescaled
//    only when a row max grows by more than 2^8; exact after the final
//    division) and round the probabilities to bf16.  Each page's probabilities
//    and per-row rescale factors are staged in shared memory in the layout the
//    value CTA's MMA reads and moved there with one bulk copy (a contiguous
//    copy runs at twice the rate of per-row remote stores; its bytes complete
//    the receiver's barrier).
//  * CTA 1, the value CTA, keeps the full 128 x 512 fp32 output in tensor
//    memory (all 512 columns), streams the 512 latent dims of the same pages
//    in half-page units through a 3-deep ring (the second read of a page is
//    an L2 hit) and accumulates O += P . V with tcgen05.mma (A = P from shared
//    memory, B = V MN-major, N = 256 per half).  The probabilities arrive in
//    a ring of six 18 KB units (one per page, two when the page also sends
//    the low bf16 parts of its probabilities).  Four warps apply row rescales
//    and zero the rows of a last page past the sequence end (0 x NaN would
//    poison O); eight warps write the normalised output with TMA tensor
//    stores (or the split's partial output, merged later).
//  * Each worker takes a contiguous range of the cost-weighted split
//    partition (common.cuh): work items are (sequence, row group, page
//    range), planned on the device in batches of up to 64.
// The data flow is one-way (score CTA -> value CTA), so the distributed-
// shared-memory latency is pipelined, never on a round trip.
// Every mbarrier wait is bounded (2 s): on expiry the kernel records
// MLA_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int kThreads = 320;            // 10 warps
constexpr int kRows = 128;               // query rows per work item (one row group)
constexpr int kBox = 8192;               // 64 tokens x 64 dims x bf16
constexpr int kCell = 2 * kBox;          // score CTA: box c of both pages of a pair
constexpr int kCells = 6;                // score CTA: ring depth (cells); measured on B300:
                                         // 6 is best (8: 1% slower, 4: 3% slower)
constexpr int kVUnit = 4 * kBox;         // value CTA: 256 latent dims of one page
constexpr int kVUnits = 3;               // value CTA: ring depth (half pages)
constexpr int kPBytes = kRows * 64 * 2;  // bf16 probabilities of one page (K-major, SW128)
constexpr int kInfoBytes = 16 + kRows * 8;       // header + (alpha, l) per row
constexpr int kPMsgBytes = kPBytes + kInfoBytes; // bytes delivered per page (one bulk copy)
// Probability messages travel in 18 KB units: a page takes one unit (its bf16
// probabilities, header and per-row factors) or two (then the second one
// carries the low bf16 parts).  Both CTAs advance the same unit counter.
constexpr int kPUnitBytes = 18432;
constexpr int kPUnits = 6;               // units in the value CTA's ring
constexpr int kStgPageBytes = 2 * kPUnitBytes;   // score CTA staging per page (hi unit, lo unit)
// shared-memory map (offsets from the 1 KB aligned base)
constexpr int kOffQr = 0;                // score CTA: rotary query, 128 x 64 bf16 (K-major SW128)
constexpr int kOffStg = 16384;           // score CTA: the step's two outgoing page messages
constexpr int kOffCells = kOffStg + 2 * kStgPageBytes;   // score CTA: the cells
constexpr int kOffV = 0;                 // value CTA: 3 half-page units
constexpr int kOffP = kVUnits * kVUnit;  // value CTA: probability slots (score CTA writes them)
constexpr int kScoreSmem = kOffCells + kCells * kCell;
constexpr int kValueSmem = kOffP + kPUnits * kPUnitBytes;
constexpr int kSmemBytes = (kScoreSmem > kValueSmem ? kScoreSmem : kValueSmem) + 1024;
constexpr int kMaxItems = 64;            // work items planned per batch
// TMEM columns (score CTA): score buffers 2 x 128 at [0, 256), latent query at [256, 512)
constexpr uint32_t kTmemQ = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// header flag bits of a page message
constexpr uint32_t kFlagRescale = 1u;    // rows rescaled before this page's value MMA
constexpr uint32_t kFlagLo = 2u;         // the low bf16 parts of the probabilities follow
constexpr uint64_t kWaitNs = 2000000000ull;

static_assert(kPMsgBytes <= kPUnitBytes, "probability unit too small");
static_assert(kPMsgBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
static_assert(kOffCells % 1024 == 0, "SW128 operands need 1 KB alignment");
static_assert(kOffP % 1024 == 0 && kPUnitBytes % 1024 == 0, "SW128 operands need 1 KB alignment");
static_assert(8 * 2048 <= kPBytes, "epilogue staging lives in a probability slot");
static_assert(4 * 4096 <= kPBytes, "four epilogue boxes fit in a unit's probability area");

struct Item {
  int b, j0, j1;            // sequence, page range [j0, j1)
  int g, vb;                // row group, virtual sequence b * G + g
  int w_first, w_last;      // workers holding the virtual sequence's first and last page
  int flags;                // bit 0: this worker holds the whole (virtual) sequence
};

struct SmemCtl {
  // score CTA
  uint64_t cell_full[kCells], cell_empty[kCells];
  uint64_t s_full[2], s_free[2];
  uint64_t q_ready, pfree[kPUnits];
  // value CTA
  uint64_t v_full[kVUnits], v_empty[kVUnits];
  uint64_t p_recv[kPUnits];    // a unit's bytes arrived
  uint64_t pv_done[kPUnits];   // value MMAs of the page whose first unit sits here completed
  uint64_t resc_done, vz_done;
  uint64_t o_free;          // the epilogue has read O: the next item may overwrite it
  uint64_t epi_go;          // O of the item is final (value row warps -> other warps)
  uint64_t epi_done;        // all epilogue warps are done with the staging slot
  uint64_t rows_seen[kPUnits];  // all row warps have read the header and factors in a unit
  // both
  uint64_t grp, mma_final;
  uint32_t tmem_base;
  int abort;
  int never;                // stays 0: abort flag for the final drain waits
  int n_batch, n_total;
  int scan[kThreads / 32];
  float rowx[2][kRows];     // score CTA: per-half row maxima of a step
  float rowl[2][kRows];     // score CTA: per-half row sums (last step of an item)
  // score CTA: header flags of a page, indexed by page mod 2 x slots: a word
  // is reset by the leader after the step that sent it and written again three
  // steps later, so the two never race
  uint32_t pflags[6];
  uint32_t epi_unit;        // value CTA: first unit of the item's last page (for the epilogue)
  Item items[kMaxItems];
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int pages_of(int L, int T_q, int cap) {
  return (L >= T_q && L <= cap) ? (L + kPage - 1) / kPage : 0;
}

// exclusive scan over the CTA
__device__ int cta_excl_scan(int v, int* scan, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scan[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) {
    int t = scan[i];
    if (i < warp) base += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

// Plan the work items of worker w with item index in [offset, offset + kMaxItems).
// Same partition as the CUDA-core kernel (see part_begin / part_pages), with
// the item cost the launcher chose for this kernel.
__device__ void plan_batch(const DecodeArgs& a, int w, int offset, SmemCtl* ctl) {
  const int tid = threadIdx.x;
  const int cap = a.max_blocks * kPage;
  const int C = a.item_cost;
  const int nv = a.B * a.G;   // virtual sequences (sequence, row group), b-major
  int mine = 0;
  for (int v = tid; v < nv; v += kThreads) {
    const int P = pages_of(a.seqlens[v / a.G], a.T_q, cap);
    mine += P > 0 ? C + P : 0;
  }
  int total;
  cta_excl_scan(mine, ctl->scan, &total);
  const long long U = total;
  const int Wa = part_active(U, a.W, C);
  int n_total = 0, n_batch = 0;
  if (U > 0 && w < Wa) {
    const long long x0 = part_begin(U, Wa, w), x1 = part_begin(U, Wa, w + 1);
    long long base = 0;
    int count = 0;
    for (int c0 = 0; c0 < nv && base < x1; c0 += kThreads) {
      const int v = c0 + tid;
      const int b = v < nv ? v / a.G : 0;
      const int P = v < nv ? pages_of(a.seqlens[b], a.T_q, cap) : 0;
      int chunk_total;
      const int excl = cta_excl_scan(P > 0 ? C + P : 0, ctl->scan, &chunk_total);
      const long long A = base + excl + C;   // unit of the sequence's first page
      int j0, j1;
      part_pages(x0, x1, A, P, &j0, &j1);
      const int hit = (P > 0 && j1 > j0) ? 1 : 0;
      int hits;
      const int idx = count + cta_excl_scan(hit, ctl->scan, &hits);
      if (hit && idx >= offset && idx < offset + kMaxItems) {
        Item it;
        it.b = b;
        it.g = v - b * a.G;
        it.vb = v;
        it.j0 = j0;
        it.j1 = j1;
        it.w_first = part_worker_of(U, Wa, A);
        it.w_last = part_worker_of(U, Wa, A + P - 1);
        it.flags = (j0 == 0 && j1 == P) ? 1 : 0;
        ctl->items[idx - offset] = it;
      }
      count += hits;
      base += chunk_total;
    }
    n_total = count;
    n_batch = min(kMaxItems, max(0, count - offset));
  }
  if (tid == 0) {
    ctl->n_total = n_total;
    ctl->n_batch = n_batch;
  }
  __syncthreads();
}

__device__ __forceinline__ void fail(SmemCtl* ctl, unsigned* err) {
  ctl->abort = 1;
  atomicOr(err, kErrTimeout);
}

// every lane of the warp waits; true only if all of them saw the phase complete
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, kWaitNs));
}

// the same, with acquire at cluster scope (bytes or arrivals from the peer CTA)
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, abort, kWaitNs));
}

// barrier among the warps of a role, with a bounded wait (a plain bar.sync
// could not give up if a warp left after a timeout)
__device__ __forceinline__ bool group_sync(uint64_t* grp, uint32_t& phase, volatile int* abort) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(grp);
  const bool done = warp_wait(grp, phase & 1, abort);
  ++phase;
  return done;
}

__device__ __forceinline__ uint32_t lo_half_f(uint32_t u) { return u << 16; }
__device__ __forceinline__ uint32_t hi_half_f(uint32_t u) { return u & 0xffff0000u; }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_pool,
                 const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_ws) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pslots = smem + kOffP;                  // value CTA: probability slots

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();         // 0: score CTA, 1: value CTA
  const int w = (int)cluster_id_x();
  volatile int* abort_flag = &ctl.abort;

  if (threadIdx.x == 0) {
    ctl.abort = 0;
    ctl.never = 0;
    for (int i = 0; i < kCells; ++i) {
      mbar_init(&ctl.cell_full[i], 1);
      mbar_init(&ctl.cell_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.s_free[i], 8);
    }
    for (int i = 0; i < kVUnits; ++i) {
      mbar_init(&ctl.v_full[i], 1);
      mbar_init(&ctl.v_empty[i], 1);
    }
    for (int i = 0; i < kPUnits; ++i) {
      mbar_init(&ctl.pfree[i], 1);
      mbar_init(&ctl.p_recv[i], 1);
      mbar_init(&ctl.pv_done[i], 1);
      mbar_init(&ctl.rows_seen[i], 4);
      ctl.pflags[i] = 0;
    }
    mbar_init(&ctl.q_ready, 8);
    mbar_init(&ctl.resc_done, 4);
    mbar_init(&ctl.vz_done, 4);
    mbar_init(&ctl.o_free, 8);
    mbar_init(&ctl.epi_go, 4);
    mbar_init(&ctl.epi_done, 8);
    mbar_init(&ctl.grp, 8);
    mbar_init(&ctl.mma_final, 1);
    if (rank == 1)     // the first pages' probabilities will arrive
      for (int i = 0; i < kPUnits; ++i) mbar_arrive_expect_tx(&ctl.p_recv[i], kPMsgBytes);
    fence_mbar_init_cluster();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm_pool);
  if (warp == 1) tmem_alloc(&ctl.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();   // the peer's barriers are initialised before any remote access
  cluster_wait();
  const uint32_t tmem = ctl.tmem_base;

  const float sl2 = a.scale * kLog2e;
  const int rows = a.T_q * a.H;   // query rows of a sequence (a work item takes
                                  // the <= 128 rows of one row group; the MMAs
                                  // always run 128 rows, the rest are zero padding)
  const int cap = a.max_blocks * kPage;

  uint32_t g_prod = 0, g_issue = 0;    // producer: cells (score) or units (value) issued
  uint32_t g_cell = 0;                 // score MMA: cells consumed
  uint32_t g_step = 0;                 // score CTA: page-pair steps (MMA and softmax)
  uint32_t g_page = 0;                 // pages (score softmax, value MMA and warps)
  uint32_t it_cnt = 0;                 // items (MMA issuers, value warps)
  uint32_t grp_phase = 0, n_resc = 0, n_vz = 0;
  // probability-unit counters: they run on across planning batches, like the
  // mbarrier phases they index
  uint32_t un = 0;                     // value MMA: units consumed
  uint32_t un_s = 0;                   // score leader: units sent
  // value row warps: units seen, and per unit slot the parity of the next
  // phase of its page barriers (pv_done, rows_seen advance only when the slot
  // holds a page's first unit)
  uint32_t un_v = 0, pvpar = 0, prev_slot = 0, prev_par = 0;

  for (int offset = 0;; offset += kMaxItems) {
    plan_batch(a, w, offset, &ctl);
    const int n_items = ctl.n_batch;
    if (n_items == 0) break;

    if (warp == 0) {
      // ============================================================ producer
      // (the whole warp walks the loop; lane 0 issues barriers and copies)
      const uint64_t pol = policy_evict_first();
      for (int ii = 0; ii < n_items; ++ii) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const Item it = ctl.items[ii];
        for (int jb = it.j0; jb < it.j1; jb += 32) {
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
          const int jj = jb + lane;
          int blk = -1;
          if (jj < it.j1) blk = a.block_table[(size_t)it.b * a.max_blocks + jj];
          const int nj = min(32, it.j1 - jb);
          if (rank == 0) {
            // page pairs (pairs start at j0, so they never straddle a 32-page chunk)
            for (int k = 0; k < nj; k += 2) {
              const bool two = k + 1 < nj;
              const int bA = __shfl_sync(0xffffffffu, blk, k);
              const int bB = __shfl_sync(0xffffffffu, blk, two ? k + 1 : k);
              if (lane == 0) {
                const bool okA = bA >= 0 && bA < a.num_blocks;
                const bool okB = bB >= 0 && bB < a.num_blocks;
                if (!okA || (two && !okB)) atomicOr(a.err, kErrBadIndex);
                // an invalid block is read past the pool's end: TMA fills zeros
                const int yA = okA ? bA * kPage : a.num_blocks * kPage;
                const int yB = okB ? bB * kPage : a.num_blocks * kPage;
                for (int c = 0; c < 9; ++c) {
                  if (*abort_flag) break;
                  const uint32_t sl = g_prod % kCells;
                  if (g_prod >= (uint32_t)kCells &&
                      !mbar_wait(&ctl.cell_empty[sl], ((g_prod / kCells) - 1) & 1, abort_flag, kWaitNs)) {
                    fail(&ctl, a.err);
                    break;
                  }
                  uint8_t* dst = smem + kOffCells + sl * kCell;
                  mbar_arrive_expect_tx(&ctl.cell_full[sl], two ? kCell : kBox);
                  tma_load_2d(dst, &tm_pool, &ctl.cell_full[sl], 64 * c, yA, pol);
                  if (two) tma_load_2d(dst + kBox, &tm_pool, &ctl.cell_full[sl], 64 * c, yB, pol);
                  ++g_prod;
                  ++g_issue;
                }
              }
              __syncwarp();
            }
          } else {
            for (int k = 0; k < nj; ++k) {
              const int bk = __shfl_sync(0xffffffffu, blk, k);
              if (lane == 0) {
                const bool valid = bk >= 0 && bk < a.num_blocks;
                const int y = valid ? bk * kPage : a.num_blocks * kPage;
                for (int nh = 0; nh < 2; ++nh) {
                  if (*abort_flag) break;
                  const uint32_t sl = g_prod % kVUnits;
                  if (g_prod >= (uint32_t)kVUnits &&
                      !mbar_wait(&ctl.v_empty[sl], ((g_prod / kVUnits) - 1) & 1, abort_flag, kWaitNs)) {
                    fail(&ctl, a.err);
                    break;
                  }
                  uint8_t* dst = smem + kOffV + sl * kVUnit;
                  mbar_arrive_expect_tx(&ctl.v_full[sl], kVUnit);
                  for (int bx = 0; bx < 4; ++bx)
                    tma_load_2d(dst + bx * kBox, &tm_pool, &ctl.v_full[sl], 64 * (4 * nh + bx), y, pol);
                  ++g_prod;
                  ++g_issue;
                }
              }
              __syncwarp();
            }
          }
        }
      }
    } else if (warp == 1) {
      // ============================================================ MMA issuer
      if (lane == 0) {
        if (rank == 0) {
          const uint32_t idS2 = idesc_bf16_f32(128, 128, 0, 0);
          const uint32_t idS1 = idesc_bf16_f32(128, 64, 0, 0);
          const uint8_t* qr = smem + kOffQr;
          for (int ii = 0; ii < n_items && !*abort_flag; ++ii) {
            const Item it = ctl.items[ii];
            const int n = it.j1 - it.j0;
            bool ok = mbar_wait(&ctl.q_ready, it_cnt & 1, abort_flag, kWaitNs);
            for (int k = 0; ok && k < n; k += 2) {
              const uint32_t sb = g_step & 1;
              const uint32_t id = (k + 1 < n) ? idS2 : idS1;
              if (g_step >= 2) ok = mbar_wait(&ctl.s_free[sb], ((g_step >> 1) - 1) & 1, abort_flag, kWaitNs);
              for (int c = 0; ok && c < 9; ++c) {
                const uint32_t sl = g_cell % kCells;
                ok = mbar_wait(&ctl.cell_full[sl], (g_cell / kCells) & 1, abort_flag, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* cp = smem + kOffCells + sl * kCell;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const int kk = 4 * c + q;
                  const uint64_t bd = sdesc_sw128(smem_u32(cp + q * 32), 16, 1024);
                  if (c < 8)
                    mma_ts(tmem + sb * 128, tmem + kTmemQ + kk * 8, bd, id, kk > 0);
                  else
                    mma_ss(tmem + sb * 128, sdesc_sw128(smem_u32(qr + q * 32), 16, 1024), bd, id, 1);
                }
                mma_commit(&ctl.cell_empty[sl]);
                ++g_cell;
              }
              if (!ok) break;
              mma_commit(&ctl.s_full[sb]);
              ++g_step;
            }
            if (!ok) { fail(&ctl, a.err); break; }
            ++it_cnt;
          }
        } else {
          const uint32_t idPV = idesc_bf16_f32(128, 256, 0, 1);
          for (int ii = 0; ii < n_items && !*abort_flag; ++ii) {
            const Item it = ctl.items[ii];
            const int L = a.seqlens[it.b];
            const int Pb = pages_of(L, a.T_q, cap);
            // the previous item's epilogue must have read O before it is overwritten
            bool ok = it_cnt == 0 || mbar_wait(&ctl.o_free, (it_cnt - 1) & 1, abort_flag, kWaitNs);
            for (int i = 0; ok && i < it.j1 - it.j0; ++i) {
              const uint32_t g = g_page + i, slot = un % kPUnits;
              const int j = it.j0 + i;
              ok = mbar_wait_cluster(&ctl.p_recv[slot], (un / kPUnits) & 1, abort_flag, kWaitNs);
              if (!ok) break;
              fence_proxy_async_smem();
              const uint8_t* ps = pslots + slot * kPUnitBytes;
              const uint32_t flags = *reinterpret_cast<const volatile uint32_t*>(ps + kPBytes);
              if ((flags & 1u) && i > 0) {          // rows rescaled by the value warps
                ok = mbar_wait(&ctl.resc_done, n_resc & 1, abort_flag, kWaitNs);
                ++n_resc;
              }
              if (ok && j == Pb - 1 && (L & (kPage - 1)) != 0) {   // tail rows zeroed
                ok = mbar_wait(&ctl.vz_done, n_vz & 1, abort_flag, kWaitNs);
                ++n_vz;
              }
              const bool lo = (flags & kFlagLo) != 0;
              const uint8_t* pl = pslots + ((un + 1) % kPUnits) * kPUnitBytes;   // low parts' unit
              if (ok && lo) {
                ok = mbar_wait_cluster(&ctl.p_recv[(un + 1) % kPUnits], ((un + 1) / kPUnits) & 1, abort_flag, kWaitNs);
                fence_proxy_async_smem();
              }
              for (int nh = 0; ok && nh < 2; ++nh) {
                const uint32_t u = 2 * g + nh, vs = u % kVUnits;
                ok = mbar_wait(&ctl.v_full[vs], (u / kVUnits) & 1, abort_flag, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                const uint8_t* vp = smem + kOffV + vs * kVUnit;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {   // 64 tokens, K-step 16
                  const uint64_t ad = sdesc_sw128(smem_u32(ps + kk * 32), 16, 1024);
                  const uint64_t bd = sdesc_sw128(smem_u32(vp + kk * 2048), kBox, 1024);
                  mma_ss(tmem + nh * 256, ad, bd, idPV, (i > 0 || kk > 0) ? 1 : 0);
                }
                if (lo) {
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk) {   // the same V rows, A = low parts
                    const uint64_t ad = sdesc_sw128(smem_u32(pl + kk * 32), 16, 1024);
                    const uint64_t bd = sdesc_sw128(smem_u32(vp + kk * 2048), kBox, 1024);
                    mma_ss(tmem + nh * 256, ad, bd, idPV, 1);
                  }
                }
                mma_commit(&ctl.v_empty[vs]);
              }
              if (!ok) break;
              mma_commit(&ctl.pv_done[slot]);
              un += lo ? 2 : 1;
            }
            if (!ok) { fail(&ctl, a.err); break; }
            g_page += it.j1 - it.j0;
            ++it_cnt;
          }
        }
      }
      __syncwarp();
    } else if (rank == 0) {
      // ============================================================ softmax (score CTA)
      // warp w: TMEM lane quarter w & 3 (32 rows); half 0 (warps 2-5) takes the
      // first page of each pair, half 1 (warps 6-9) the second
      const int q4 = warp & 3;
      const int half = warp >= 6 ? 1 : 0;
      const int r = 32 * q4 + lane;
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const uint32_t peer_p = mapa(smem_u32(pslots), 1);               // value CTA's slots
      const uint32_t peer_precv = mapa(smem_u32(&ctl.p_recv[0]), 1);   // + 8 * slot
      const bool leader = threadIdx.x == 64;
      uint8_t* qr = smem + kOffQr;
      for (int ii = 0; ii < n_items; ++ii) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        const Item it = ctl.items[ii];
        const int L = a.seqlens[it.b];
        const int rb = kRows * it.g;                   // first row of the group
        const int rows_g = min(kRows, rows - rb);       // its real rows
        const int t = (rb + r) / a.H;                  // query token of this row
        // padding rows (r >= rows_g) see no token at all
        const int lim = r >= rows_g ? -1 : a.causal ? (L - a.T_q + t) : (L - 1);
        const int n = it.j1 - it.j0;
        // the query row: latent dims -> TMEM (half 0: [0, 256), half 1: [256, 512)),
        // rotary dims -> shared memory (K-major SW128; half h: 16-byte chunks 4h..4h+3)
        {
          const bool real = r < rows_g;
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(a.q) + ((size_t)it.b * rows + rb + (real ? r : 0)) * a.D);
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 x = real ? __ldg(src + half * 32 + c * 8 + u) : make_uint4(0u, 0u, 0u, 0u);
              v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
            }
            tmem_st32(tmem + lane_off + kTmemQ + half * 128 + 32 * c, v);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = 4 * half + c;
            *reinterpret_cast<uint4*>(qr + r * 128 + ((ch ^ (r & 7)) << 4)) =
                real ? __ldg(src + 64 + ch) : make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.q_ready);
        }
        float m_run = -INFINITY, l_half = 0.f;
        bool ok = true;
        for (int k = 0; k < n; k += 2) {
          const bool two = k + 1 < n;
          const bool has = half == 0 || two;           // this half's page exists
          const uint32_t sb = g_step & 1;
          const uint32_t gA = g_page;
          const int jh = it.j0 + k + half;
          const bool last_step = k + 2 >= n;
          int bk = -1;
          if (has) bk = __ldg(a.block_table + (size_t)it.b * a.max_blocks + jh);
          const bool page_ok = has && bk >= 0 && bk < a.num_blocks;
          if (!warp_wait(&ctl.s_full[sb], (g_step >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          float x[64];
          tmem_ld64(tmem + lane_off + sb * 128 + 64 * half, x);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.s_free[sb]);     // score buffer reusable
          // mask (tokens past the visible range, a missing page, a bad block id)
          const int tok0 = jh * kPage;
          if (!page_ok || tok0 + 63 > L - a.T_q || r >= rows_g) {
            const int lim_page = page_ok ? lim : -1;
#pragma unroll
            for (int q = 0; q < 64; ++q) x[q] = (tok0 + q <= lim_page) ? x[q] : -INFINITY;
          }
          float mx = x[0];
#pragma unroll
          for (int q = 1; q < 64; ++q) mx = fmaxf(mx, x[q]);
          ctl.rowx[half][r] = mx;
          const uint32_t fh = (gA + half) % 6;   // this half's page flags
          {
            // Precision of the bf16 probabilities: a page whose largest
            // probability is not small against the row sum so far also sends
            // the low bf16 parts (p - bf16(p)).  Tested conservatively, before
            // the rows' maxima are merged: against this half's own running sum
            // and the previous reference (both can only make the test pass more
            // often than with the merged values).
            // The item's last page always sends them: its two units then give
            // the value CTA's epilogue its staging space.
            const bool heavy = has && ex2(mx * sl2 - m_run) >= l_half;
            const bool item_last = has && last_step && half == (two ? 1 : 0);
            if ((__any_sync(0xffffffffu, heavy) || item_last) && lane == 0) atomicOr(&ctl.pflags[fh], kFlagLo);
          }
          if (leader) bulk_wait_read0();   // the previous step's copies have read the staging
          if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }   // [A]
          const float m_page = fmaxf(mx, ctl.rowx[half ^ 1][r]) * sl2;
          const float m_new = fmaxf(m_run, m_page);
          const bool need = m_new > m_run + kRescaleThreshold;
          float alpha = 1.f;
          if (need) {
            alpha = ex2(m_run - m_new);     // 0 when m_run = -inf
            m_run = m_new;
            l_half *= alpha;
          }
          uint8_t* stg = smem + kOffStg + half * kStgPageBytes;   // this half's page message
          if (has) {
            // probabilities, rounded to bf16 (and, for a heavy page, the
            // residual rounded again); l sums exactly what the value MMA sees.
            // Rows are staged in the layout the value CTA's MMA reads
            // (K-major SW128: 16-byte chunk c of row r at c ^ (r & 7)).
            const bool lo = (ctl.pflags[fh] & kFlagLo) != 0;
            float psum = 0.f;
            const float neg_m = -m_run;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t pk[4], pl[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x0 = x[8 * c + 2 * e], x1 = x[8 * c + 2 * e + 1];
                const float p0 = x0 == -INFINITY ? 0.f : ex2(fmaf(x0, sl2, neg_m));
                const float p1 = x1 == -INFINITY ? 0.f : ex2(fmaf(x1, sl2, neg_m));
                pk[e] = pack_bf16x2(p0, p1);
                const float h0 = __uint_as_float(lo_half_f(pk[e])), h1 = __uint_as_float(hi_half_f(pk[e]));
                psum += h0 + h1;
                if (lo) {
                  pl[e] = pack_bf16x2(p0 - h0, p1 - h1);
                  psum += __uint_as_float(lo_half_f(pl[e])) + __uint_as_float(hi_half_f(pl[e]));
                }
              }
              const int off = r * 128 + ((c ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(stg + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              if (lo) *reinterpret_cast<uint4*>(stg + kPUnitBytes + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            l_half += psum;
          }
          if (__any_sync(0xffffffffu, need) && k > 0 && lane == 0 && half == 0)
            atomicOr(&ctl.pflags[gA % 6], kFlagRescale);
          float l_tot = 0.f;
          if (last_step) {
            ctl.rowl[half][r] = l_half;
            if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }
            l_tot = ctl.rowl[0][r] + ctl.rowl[1][r];
            if (half == 0 && r < rows_g) {
              const float lse = l_tot > 0.f ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
              const int wslot = it.vb + w;
              if (it.flags & 1) { if (a.lse) a.lse[(size_t)it.b * rows + rb + r] = lse; }
              else a.ws_lse[(size_t)wslot * a.SR + r] = lse;
              if (r == 0 && it.j0 == 0) a.meta[it.vb] = make_int2(it.w_first, it.w_last);
            }
          }
          // per-row (alpha, l): the rescale factor rides on the pair's first
          // page; l (the row sum) on the item's last page
          if (has) {
            const bool last_page = last_step && half == (two ? 1 : 0);
            *reinterpret_cast<float2*>(stg + kPBytes + 16 + r * 8) =
                make_float2(half == 0 ? alpha : 1.f, last_page ? l_tot : 0.f);
            fence_proxy_async_smem();      // the bulk copy reads the staging
          }
          if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }   // [B]
          // headers (flags gathered from all warps of each page), then per unit
          // one bulk copy into the value CTA's ring once the value CTA has freed
          // that unit; its bytes complete the unit's barrier there.  Only this
          // thread waits here: the staging is local, so the softmax of the
          // next step runs while the value CTA catches up.
          if (leader) {
            bool fr = true;
            for (uint32_t e = 0; e < (two ? 2u : 1u) && fr; ++e) {
              uint8_t* st = smem + kOffStg + e * kStgPageBytes;
              const uint32_t fi = (gA + e) % 6;
              const uint32_t fl = ctl.pflags[fi];
              ctl.pflags[fi] = 0u;              // ready for page gA + e + 6
              *reinterpret_cast<uint4*>(st + kPBytes) = make_uint4(fl, 0u, 0u, 0u);
              fence_proxy_async_smem();
              for (uint32_t part = 0; part < ((fl & kFlagLo) ? 2u : 1u) && fr; ++part) {
                const uint32_t ui = un_s++, us = ui % kPUnits;
                if (ui >= (uint32_t)kPUnits)
                  fr = mbar_wait_cluster(&ctl.pfree[us], ((ui / kPUnits) - 1) & 1, abort_flag, kWaitNs);
                if (fr)
                  bulk_copy_to_peer(peer_p + us * kPUnitBytes, st + part * kPUnitBytes, kPMsgBytes,
                                    peer_precv + 8 * us);
              }
            }
            bulk_commit();
            if (!fr) fail(&ctl, a.err);
          }
          g_page += two ? 2 : 1;
          ++g_step;
        }
        if (!ok) { fail(&ctl, a.err); break; }
      }
    } else {
      // ============================================================ value CTA warps
      // warps 2-5 ("row warps"): page bookkeeping, row rescales, tail zeroing;
      // all eight: the epilogue, warp w writing rows 32 (w & 3) .. + 31 and
      // output columns [256 * (w >= 6), + 256)
      const int q4 = warp & 3;
      const int ch = warp >= 6 ? 1 : 0;
      const bool row_warp = warp < 6;
      const int r = 32 * q4 + lane;
      const int tq = threadIdx.x - 64;             // 0..127 (row warps)
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const uint32_t peer_pfree = mapa(smem_u32(&ctl.pfree[0]), 0);   // + 8 * unit slot
      for (int ii = 0; ii < n_items; ++ii) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        const Item it = ctl.items[ii];
        const int L = a.seqlens[it.b];
        const int Pb = pages_of(L, a.T_q, cap);
        const int n = it.j1 - it.j0;
        bool ok = true;
        if (row_warp) {
          for (int i = 0; i < n; ++i) {
            const uint32_t g = g_page + i, slot = un_v % kPUnits;
            const int j = it.j0 + i;
            uint8_t* ps = pslots + slot * kPUnitBytes;
            if (!warp_wait_cluster(&ctl.p_recv[slot], (un_v / kPUnits) & 1, abort_flag)) { ok = false; break; }
            const uint32_t flags = *reinterpret_cast<const volatile uint32_t*>(ps + kPBytes);
            const bool lo = (flags & kFlagLo) != 0;
            const uint32_t par = (pvpar >> slot) & 1;
            const float* info = reinterpret_cast<const float*>(ps + kPBytes + 16);
            if (j == Pb - 1 && (L & (kPage - 1)) != 0) {
              // last page: zero the V rows past the sequence end (they may hold NaN)
              const int nv = L & (kPage - 1);
              const int per_box = (kPage - nv) * 8;    // 16-byte chunks per box
              for (int nh = 0; nh < 2 && ok; ++nh) {
                const uint32_t u = 2 * g + nh, vs = u % kVUnits;
                if (!warp_wait(&ctl.v_full[vs], (u / kVUnits) & 1, abort_flag)) { ok = false; break; }
                uint4* vp = reinterpret_cast<uint4*>(smem + kOffV + vs * kVUnit);
                for (int q = tq; q < 4 * per_box; q += kRows) {
                  const int bx = q / per_box, rem = q - bx * per_box;
                  vp[(bx * kBox + (nv + rem / 8) * 128) / 16 + (rem & 7)] = make_uint4(0, 0, 0, 0);
                }
              }
              if (!ok) break;
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl.vz_done);
            }
            if ((flags & 1u) && i > 0) {
              // rescale O rows before this page's value MMA: O holds pages < j
              if (!warp_wait(&ctl.pv_done[prev_slot], prev_par, abort_flag)) { ok = false; break; }
              tc_fence_after();
              const float alpha = info[2 * r];
#pragma unroll 1
              for (int c = 0; c < 8; ++c) {
                float o[64];
                tmem_ld64(tmem + lane_off + 64 * c, o);
                tmem_ld_wait();
                uint32_t u0[32], u1[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                  u0[q] = __float_as_uint(o[q] * alpha);
                  u1[q] = __float_as_uint(o[32 + q] * alpha);
                }
                tmem_st32(tmem + lane_off + 64 * c, u0);
                tmem_st32(tmem + lane_off + 64 * c + 32, u1);
              }
              tmem_st_wait();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl.resc_done);
            }
            // header and factors read by this warp (one barrier per unit slot: a
            // warp cannot reach the slot's next page before this unit is released)
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.rows_seen[slot]);
            // this page's value MMA done
            if (!warp_wait(&ctl.pv_done[slot], par, abort_flag)) { ok = false; break; }
            if (i < n - 1) {
              // the page's units may be refilled once every row warp is past its header
              if (threadIdx.x == 64) {
                if (mbar_wait(&ctl.rows_seen[slot], par, abort_flag, kWaitNs)) {
                  for (uint32_t e = 0; e < (lo ? 2u : 1u); ++e) {
                    const uint32_t us = (un_v + e) % kPUnits;
                    mbar_arrive_expect_tx(&ctl.p_recv[us], kPMsgBytes);
                    mbar_arrive_remote(peer_pfree + 8 * us);
                  }
                } else {
                  fail(&ctl, a.err);
                }
              }
              __syncwarp();
            } else {
              // O is final; the last page's two units (it always carries low
              // parts) become the epilogue staging and are handed back after it
              if (threadIdx.x == 64) ctl.epi_unit = lo ? un_v : 0xffffffffu;
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl.epi_go);
            }
            prev_slot = slot;
            prev_par = par;
            pvpar ^= 1u << slot;
            un_v += lo ? 2 : 1;
          }
        }
        if (ok && !warp_wait(&ctl.epi_go, it_cnt & 1, abort_flag)) ok = false;
        if (!ok) { fail(&ctl, a.err); break; }
        // ---- epilogue: normalise and write the item's 128 x 512 output, each
        // warp staging 32 rows x 16 columns at a time for full-sector writes
        tc_fence_after();
        const uint32_t eu = ctl.epi_unit;
        if (eu == 0xffffffffu) { fail(&ctl, a.err); break; }   // cannot happen: the last page sends low parts
        uint8_t* ps_last = pslots + (eu % kPUnits) * kPUnitBytes;
        uint8_t* ps_lo = pslots + ((eu + 1) % kPUnits) * kPUnitBytes;
        const float l_row = reinterpret_cast<const float*>(ps_last + kPBytes + 16)[2 * r + 1];
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        const bool whole = it.flags & 1;
        const int rb = kRows * it.g;                            // first row of the row group
        const int grp_rows = min(32, min(kRows, rows - rb) - 32 * q4);   // real rows of this warp's group
        float* out_base = (whole ? a.o + ((size_t)it.b * rows + rb) * a.d_c
                                 : a.ws_o + (size_t)(it.vb + w) * a.SR * a.d_c) + 256 * ch;
        if (grp_rows > 0) out_base += (size_t)(32 * q4) * a.d_c;
        // every thread must have read l before the staging writes below
        __syncwarp();
        if (grp_rows == 32) {
          // whole 32-row group: 32 x 32 fp32 boxes staged (SW128) in the
          // slot's probability areas (not its factors) and written by TMA
          const CUtensorMap* tmo = whole ? &tm_o : &tm_ws;
          const int row0 = (whole ? it.b * rows + rb : (it.vb + w) * a.SR) + 32 * q4;
          const int wi = warp - 2;
          uint8_t* box = wi < 4 ? ps_last + wi * 4096 : ps_lo + (wi - 4) * 4096;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_off + 256 * ch + 32 * c, o);
            tmem_ld_wait();
            if (lane == 0) bulk_wait_read0();     // the previous box has been read
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(box + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                  make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv, o[4 * k + 3] * inv);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(tmo, box, 256 * ch + 32 * c, row0);
              bulk_commit();
            }
          }
          if (lane == 0) bulk_wait_read0();         // staging free before the slot is handed back
          __syncwarp();
        }
        // a warp's own 4 KB of the two units (the same region its TMA boxes
        // would use, so a partial group never overlaps another warp's box)
        float4* stg = reinterpret_cast<float4*>((warp - 2) < 4 ? ps_last + (warp - 2) * 4096
                                                                : ps_lo + (warp - 6) * 4096);   // 32 rows x 4 float4
#pragma unroll 1
        for (int c = 0; c < (grp_rows > 0 && grp_rows < 32 ? 4 : 0); ++c) {
          float o[64];
          tmem_ld64(tmem + lane_off + 256 * ch + 64 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int sr = 0; sr < 4; ++sr) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              stg[lane * 4 + (e ^ ((lane >> 1) & 3))] =
                  make_float4(o[16 * sr + 4 * e] * inv, o[16 * sr + 4 * e + 1] * inv,
                              o[16 * sr + 4 * e + 2] * inv, o[16 * sr + 4 * e + 3] * inv);
            __syncwarp();
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
              const int row = lane / 4 + 8 * tt, e = lane & 3;
              if (row < grp_rows)
                reinterpret_cast<float4*>(out_base + (size_t)row * a.d_c + 64 * c + 16 * sr)[e] =
                    stg[row * 4 + (e ^ ((row >> 1) & 3))];
            }
            __syncwarp();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl.o_free);      // O may be overwritten now
          mbar_arrive(&ctl.epi_done);
        }
        if (threadIdx.x == 64) {
          // hand the staging slot back once every epilogue warp is done with it
          if (mbar_wait(&ctl.epi_done, it_cnt & 1, abort_flag, kWaitNs)) {
            for (uint32_t e = 0; e < 2; ++e) {
              const uint32_t us = (eu + e) % kPUnits;
              mbar_arrive_expect_tx(&ctl.p_recv[us], kPMsgBytes);
              mbar_arrive_remote(peer_pfree + 8 * us);
            }
          } else {
            fail(&ctl, a.err);
          }
        }
        __syncwarp();
        g_page += n;
        ++it_cnt;
      }
    }
    __syncthreads();
    if (*abort_flag) break;
    if (offset + kMaxItems >= ctl.n_total) break;
  }

  // the merge pass may start launching now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- drain: all MMAs complete, all TMA loads and bulk copies done, then free TMEM
  if (rank == 0 && threadIdx.x == 64) bulk_wait0();
  if (rank == 1 && warp >= 2 && lane == 0) bulk_wait0();   // output stores complete
  if (warp == 1 && lane == 0) {
    mma_commit(&ctl.mma_final);
    if (!mbar_wait(&ctl.mma_final, 0, &ctl.never, kWaitNs)) atomicOr(a.err, kErrTimeout);
  }
  if (warp == 0 && lane == 0) {
    const uint32_t nring = rank == 0 ? kCells : kVUnits;
    uint64_t* full = rank == 0 ? ctl.cell_full : ctl.v_full;
    for (uint32_t k = 0; k < nring && k < g_issue; ++k) {
      const uint32_t g = g_issue - 1 - k;
      if (!mbar_wait(&full[g % nring], (g / nring) & 1, &ctl.never, kWaitNs)) atomicOr(a.err, kErrTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  cluster_arrive();   // the peer may still target our shared memory until here
  cluster_wait();
}

CUresult (*g_encode)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                     CUtensorMapFloatOOBfill) = nullptr;

cudaError_t get_encode() {
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
  g_encode = reinterpret_cast<decltype(g_encode)>(fn);
  return cudaSuccess;
}

cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                     uint32_t box_cols, uint32_t box_rows, bool f32 = false) {
  const uint64_t es_bytes = f32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int g_max_clusters[64] = {};

}  // namespace

bool tc_supported(int dtype, int H, int T_q, int d_c, int d_r) {
  // query rows (heads x query tokens) in groups of up to 128; a short group is padded
  return dtype == BF16 && d_c == 512 && d_r == 64 && H * T_q >= 1;
}

int tc_item_cost(int rows) {
  // Fixed cost of one work item, in pages: the worker loads the item's query
  // rows through the same SM port that streams the pages, and the value CTA
  // drains 128 x 512 fp32 of output before the next item may start.  Measured
  // on B300 by sweeping the cost: about five pages' time at 128 query rows,
  // three at 32.
  return 2 + (3 * rows + 64) / 128;
}

int tc_workers(int num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (!g_max_clusters[dev]) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    g_max_clusters[dev] = n;
  }
  return g_max_clusters[dev];
}

cudaError_t tensor_map_encoder(TensorMapEncodeFn* fn) {
  const cudaError_t e = get_encode();
  if (e == cudaSuccess) *fn = g_encode;
  return e;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  if ((long long)a.num_blocks * kPage >= (1LL << 31)) return cudaErrorInvalidValue;
  CUtensorMap tm_pool, tm_o, tm_ws;
  e = make_map(&tm_pool, a.cache, (uint64_t)a.D, (uint64_t)a.num_blocks * kPage, 64, 64);
  if (e != cudaSuccess) return e;
  // outputs and split parts: [rows, 512] fp32, written in 32 x 32 boxes
  const uint64_t rows = (uint64_t)a.T_q * a.H;
  e = make_map(&tm_o, a.o, (uint64_t)a.d_c, (uint64_t)a.B * rows, 32, 32, true);
  if (e != cudaSuccess) return e;
  e = make_map(&tm_ws, a.ws_o, (uint64_t)a.d_c, ((uint64_t)a.B * a.G + a.W) * a.SR, 32, 32, true);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.W);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel, a, tm_pool, tm_o, tm_ws);
}

}  // namespace mla
