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
// How (B300-specific).  One split worker is a cluster of two CTAs on two SMs.
// The output accumulator (128 x 512 fp32) fills a whole SM's tensor memory,
// and the score side needs the query (288 columns) and score buffers in
// tensor memory, so the two halves of the work sit on different SMs:
//  * CTA 0, the score CTA, loads each 64-token page with ONE 4-D TMA copy
//    (72 KB; every copy instruction costs a fixed ~0.3-0.5 us of the SM's
//    copy engine on this part, so small boxes cannot keep up with HBM) into
//    a ring of three page slots, and keeps three pages ahead in L2 with
//    tensor prefetches.  The 4-D box lays a page out as [8-token group]
//    [64-dim chunk][8 tokens][64 dims] with 128-byte swizzle, so each
//    (group, chunk) is one 1 KB swizzle atom and an MMA operand over the
//    page's 64 tokens is a uniform stride of 9 KB.  Scores S = Q . C^T
//    (M = 128 rows, K = 576) are computed for the pages of an item in pairs
//    into adjacent tensor-memory buffers.  The ring places every pair in
//    adjacent slots, (0, 1) or (1, 2) (page_slot), so a pair is always one
//    operand of 128 tokens: 36 MMAs with N = 128, which on this part take as
//    long as 36 with N = 64.  An odd last page is one N = 64 chain.  The
//    MMAs are issued from a rolled chunk loop, which keeps the issuing code
//    small and resident in the instruction cache next to the softmax code.
//    The whole query is the A operand in tensor memory.  Two groups of four
//    softmax warps take the first and the second page of each pair (one
//    row per thread, all 64 tokens), run a base-2 online softmax
//    with a lazy running max passed from page to page (the output is rescaled
//    only when a row max grows by more than 2^8; exact after the final
//    division) and round the probabilities to bf16.  Each page's
//    probabilities and per-row info (reference max, sum of the rounded
//    probabilities) are written from registers into this worker's message
//    ring in global memory (L2), already in the layout the value CTA's MMA
//    reads: chunk-major (16-byte chunk c of row r at c * 2048 + r * 16, the
//    K-major operand layout without swizzle), so each store instruction of a
//    warp writes 512 contiguous bytes; a heavy page (a probability not small against its
//    row's running sum) also sends the low bf16 parts.  A signaler warp sends
//    the page's flags to the value CTA with one remote store and an mbarrier
//    arrive (release at cluster scope).
//  * CTA 1, the value CTA, keeps the 128 x 512 fp32 output in tensor memory.
//    Its producer loads the 512 latent dims of the same pages (two 32 KB
//    boxes per page, in flight together: one copy alone streams slowly; an L2
//    hit: the score CTA's copy marks them evict-last) into a ring of two, and
//    copies each page's message with one or two bulk copies
//    into a ring of three probability units and two low-part buffers.  The
//    MMA warp accumulates O += P . V (A = P from shared memory, B = V
//    MN-major, N = 256).  Four row warps zero the low parts of row quarters
//    that sent none, apply row rescales, keep the row sums and zero the rows
//    of a last page past the sequence end (0 x NaN would poison O); eight
//    warps write the normalised output with TMA tensor stores (or the
//    split's partial output, merged later).
//  * Each worker takes a contiguous range of the cost-weighted split
//    partition (common.cuh): work items are (sequence, row group, page
//    range), planned on the device in batches of up to 32.
// Distributed shared memory carries only flags and arrivals (it moves ~30
// GB/s per SM pair on this part); bulk data moves through L2.
// Every mbarrier wait is bounded (2 s): on expiry the kernel records
// MLA_ERR_TIMEOUT, drains its copies and MMAs, frees tensor memory and
// returns.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int kThreads = 352;            // 11 warps
constexpr int kRows = 128;               // query rows per work item (one row group)
constexpr int kPageBytes = kPage * 576 * 2;   // 73,728: one page, [tg 8][chunk 9][8][64]
constexpr int kSlots = 3;                // score CTA: page ring
constexpr int kVBytes = 65536;           // value CTA: the 512 latent dims of a page, [tg 8][chunk 8][8][64]
constexpr int kVSlots = 2;               // value CTA: ring of pages
constexpr int kPBytes = kRows * 64 * 2;  // bf16 probabilities of one page (K-major, SW128)
constexpr int kInfoBytes = kRows * 8;    // per row: the reference max of the page's probabilities and their sum
constexpr int kHiBytes = kPBytes + kInfoBytes;   // 17,408: probabilities + row info
constexpr int kHiUnits = 3;              // value CTA: units for the probabilities (page g in g % 3)
constexpr int kLoBufs = 2;               // value CTA: buffers for low parts (heavy pages)
constexpr int kMsgBytes = kHiBytes + kPBytes;    // a page's message: hi unit, then low parts
constexpr int kGSlots = 8;               // message ring: page slots per worker
constexpr int kPrefetch = 3;             // pages kept ahead in L2
constexpr int kOffV = 0;
constexpr int kOffHi = kVSlots * kVBytes;
constexpr int kOffLo = kOffHi + kHiUnits * kHiBytes;
constexpr int kScoreSmem = kSlots * kPageBytes;
constexpr int kValueSmem = kOffLo + kLoBufs * kPBytes;
constexpr int kSmemBytes = (kScoreSmem > kValueSmem ? kScoreSmem : kValueSmem) + 1024;
constexpr int kMaxItems = 32;            // work items planned per batch
// TMEM columns (score CTA): latent query [0, 256), rotary query [256, 288),
// score buffers [384, 448) (first page of a pair) and [448, 512) (second page)
constexpr uint32_t kTmemQr = 256;
constexpr uint32_t kTmemS = 384;   // the first page of a unit; the second at +64 or -64

// Ring slot of a page of the score CTA.  An item's pages go in units: a pair
// (pages k, k + 1 for even k) or an odd last page alone.  A unit's first page
// goes to slot 0 or 2 (alternating unit by unit), a pair's second page to
// slot 1: every pair then sits in adjacent slots, (0, 1) or (1, 2), and is ONE
// MMA operand of 128 tokens.  On this part an M = 128, K = 16 MMA takes as
// long at N = 64 as at N = 128, so a pair scored as two N = 64 chains costs
// twice as much per page.
__device__ __forceinline__ uint32_t page_slot(uint32_t unit, int second) {
  return second ? 1u : ((unit & 1u) ? 2u : 0u);
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// message flags: the page has low parts (bit 1); bit 4 + q: row quarter q
// wrote them (the other quarters' low parts are zero)
constexpr uint32_t kFlagLo = 2u;
constexpr uint64_t kWaitNs = 2000000000ull;

static_assert(kPageBytes % 1024 == 0 && kVBytes % 1024 == 0, "SW128 operands need 1 KB alignment");
static_assert(kOffHi % 1024 == 0 && kHiBytes % 1024 == 0 && kOffLo % 1024 == 0, "SW128 operands need 1 KB alignment");
static_assert(4 * 4096 <= kPBytes, "epilogue staging: four warps' boxes in a probability area");
static_assert(kPrefetch < 32, "the prefetch cursor looks at most one block-id chunk ahead");

}  // namespace

size_t tc_msg_bytes_per_worker() { return (size_t)kGSlots * kMsgBytes; }

namespace {

struct Item {
  int b, j0, j1;            // sequence, page range [j0, j1)
  int g, vb;                // row group, virtual sequence b * G + g
  int w_first, w_last;      // workers holding the virtual sequence's first and last page
  int flags;                // bit 0: this worker holds the whole (virtual) sequence
};

struct SmemCtl {
  // score CTA
  uint64_t slot_full[kSlots], slot_empty[kSlots];
  uint64_t s_full[2], s_free[2];   // score buffer of the first / second page of a pair
  uint64_t q_ready;
  uint64_t q_free;             // the scores of an item are complete: its query may be overwritten
  uint64_t gfree[kGSlots];     // a message slot may be rewritten (the value CTA's copies of it landed)
  uint64_t written[8];         // a softmax group wrote page g's message ([g % 8], count 4)
  // value CTA
  uint64_t v_full[kVSlots], v_empty[kVSlots];
  uint64_t p_ready[kGSlots];   // the score CTA wrote page g's message (remote arrive)
  uint64_t msg_full[kHiUnits]; // page g's message copied into unit g % 3 (and a low-part buffer)
  uint64_t vready[8];          // page g's probabilities are in shared memory, rescale and tail done
  uint64_t pv_done[8];         // value MMAs of page g completed
  uint64_t o_free;          // the epilogue has read O: the next item may overwrite it
  uint64_t epi_go;          // O of the item is final (value row warps -> other warps)
  uint64_t epi_done;        // all epilogue warps are done with the staging areas
  // both
  uint64_t mma_final;
  uint32_t pflag_in[kGSlots];  // value CTA: flags of a page (remote store by the score CTA)
  uint32_t uflag[8];           // value CTA: flags of page g at [g % 8], bit 8 its low-part buffer (producer -> row warps, MMA)
  uint32_t tmem_base;
  int abort;
  int never;                // stays 0: abort flag for the final drain waits
  int n_batch, n_total, n_flat;
  int scan[kThreads / 32];
  int item_flat[kMaxItems + 1];   // first page (in the batch's page order) of each item
  // score CTA: flags of page g at [g % 8], gathered with atomicOr; a word is
  // read and reset by the signaler after the page's `written` barrier and
  // written again eight pages later
  uint32_t pflags[8];
  // score CTA: the reference max of each row for the latest page, passed
  // between the two softmax groups: ((page index + 1) << 32) | float bits
  unsigned long long mref[kRows];
  float lrow[kRows];           // value CTA: row sums of an item (row warps -> epilogue warps)
  uint32_t epi_lo;             // value CTA: low-part buffer of the item's last page (epilogue staging)
  uint32_t epi_count;          // value CTA: items whose epilogue no longer uses its staging buffers
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
  __syncthreads();
  if (tid == 0) {
    ctl->n_total = n_total;
    ctl->n_batch = n_batch;
    int f = 0;
    for (int i = 0; i < n_batch; ++i) {
      ctl->item_flat[i] = f;
      f += ctl->items[i].j1 - ctl->items[i].j0;
    }
    ctl->item_flat[n_batch] = f;
    ctl->n_flat = f;
  }
  __syncthreads();
}

// block id of the batch's f-th page (0 <= f < n_flat)
__device__ __forceinline__ int block_of(const DecodeArgs& a, const SmemCtl* ctl, int n_items, int f) {
  int ii = 0;
  while (ii + 1 < n_items && ctl->item_flat[ii + 1] <= f) ++ii;
  const Item& it = ctl->items[ii];
  return __ldg(a.block_table + (size_t)it.b * a.max_blocks + it.j0 + (f - ctl->item_flat[ii]));
}

__device__ __forceinline__ void fail(SmemCtl* ctl, unsigned* err) {
  ctl->abort = 1;
  atomicOr(err, kErrTimeout);
}

// every lane of the warp waits; true only if all of them saw the phase complete
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t budget) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, budget));
}

// the same, with acquire at cluster scope (arrivals from the peer CTA)
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  uint64_t budget) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, abort, budget));
}

// wait until the tag (high 32 bits) of a shared-memory word is `tag`; the
// word is returned in *out (bounded like the barrier waits)
__device__ __forceinline__ bool wait_tag(const volatile unsigned long long* p, uint32_t tag,
                                         unsigned long long* out, volatile int* abort, uint64_t budget) {
  unsigned long long e = *p;
  if ((uint32_t)(e >> 32) == tag) { *out = e; return true; }
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    e = *p;
    if ((uint32_t)(e >> 32) == tag) { *out = e; return true; }
    if (*abort) return false;
    if (globaltimer_ns() - t0 > budget) return false;
  }
}

// wait until a counter in shared memory reaches v (bounded like the barrier waits)
__device__ __forceinline__ bool wait_count(const volatile uint32_t* c, uint32_t v, volatile int* abort,
                                           uint64_t budget) {
  if (*c >= v) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (*c >= v) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > budget) return false;
    __nanosleep(32);
  }
}

__device__ __forceinline__ uint32_t lo_half_f(uint32_t u) { return u << 16; }
__device__ __forceinline__ uint32_t hi_half_f(uint32_t u) { return u & 0xffff0000u; }

// The query row r of an item into tensor memory, one half of it: half 0
// the latent dims [0, 256) and rotary dims [512, 544), half 1 the latent dims
// [256, 512) and rotary dims [544, 576).  Latent dim d goes to column d / 2,
// rotary dim 512 + e to column 256 + e / 2 (bf16 pairs).  Padding rows are
// zero.  The warp arrives on `ready` when its part is in.
__device__ __forceinline__ void load_query_row(const DecodeArgs& a, const Item& it, int rows, uint32_t tmem,
                                               uint32_t lane_off, int r, int half, uint64_t* ready) {
  const int rb = kRows * it.g;
  const bool real = r < min(kRows, rows - rb);
  const uint4* src = reinterpret_cast<const uint4*>(
      static_cast<const __nv_bfloat16*>(a.q) + ((size_t)it.b * rows + rb + (real ? r : 0)) * a.D);
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int c2 = 0; c2 < 2; ++c2) {
    uint4 x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) x[u] = real ? __ldg(src + half * 32 + c2 * 16 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t v[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        v[4 * u] = x[8 * c + u].x; v[4 * u + 1] = x[8 * c + u].y;
        v[4 * u + 2] = x[8 * c + u].z; v[4 * u + 3] = x[8 * c + u].w;
      }
      tmem_st32(tmem + lane_off + half * 128 + 64 * c2 + 32 * c, v);
    }
  }
  {
    uint32_t v[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 x = real ? __ldg(src + 64 + 4 * half + u) : make_uint4(0u, 0u, 0u, 0u);
      v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
    }
    tmem_st16(tmem + lane_off + kTmemQr + 16 * half, v);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(ready);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_page,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const __grid_constant__ CUtensorMap tm_ws) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();         // 0: score CTA, 1: value CTA
  const int w = (int)cluster_id_x();
  volatile int* abort_flag = &ctl.abort;
  const uint64_t wait_ns = a.wait_ns ? a.wait_ns : kWaitNs;
  // this worker's message ring: page g in slot g % kGSlots
  unsigned char* gmsg = a.msg + (size_t)w * kGSlots * kMsgBytes;

  if (threadIdx.x == 0) {
    ctl.abort = 0;
    ctl.never = 0;
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&ctl.slot_full[i], 1);
      mbar_init(&ctl.slot_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.s_free[i], 4);
    }
    for (int i = 0; i < kGSlots; ++i) {
      mbar_init(&ctl.gfree[i], 1);
      mbar_init(&ctl.p_ready[i], 1);
      ctl.pflag_in[i] = 0;
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(&ctl.v_full[i], 1);
      mbar_init(&ctl.v_empty[i], 1);
    }
    for (int i = 0; i < kHiUnits; ++i) mbar_init(&ctl.msg_full[i], 1);
    ctl.epi_count = 0;
    for (int i = 0; i < 8; ++i) {
      mbar_init(&ctl.written[i], 4);
      mbar_init(&ctl.vready[i], 4);
      mbar_init(&ctl.pv_done[i], 1);
      ctl.pflags[i] = 0;
    }
    for (int i = 0; i < kRows; ++i) ctl.mref[i] = 0ull;
    mbar_init(&ctl.q_ready, 8);
    mbar_init(&ctl.q_free, 1);
    mbar_init(&ctl.o_free, 8);
    mbar_init(&ctl.epi_go, 4);
    mbar_init(&ctl.epi_done, 8);
    mbar_init(&ctl.mma_final, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_page);
    tma_prefetch_desc(&tm_v);
  }
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

  uint32_t g_prod = 0;                 // producer: pages walked
  uint32_t g_issue = 0;                // producer: score CTA: 1 + last page loaded; value CTA: pages loaded
  uint32_t g_page = 0;                 // pages (MMA issuers, softmax, value warps)
  uint32_t g_unit = 0;                 // score CTA: page units (producer, MMA issuer, softmax)
  // score CTA: pages put in (producer) or taken from (MMA issuer) each ring
  // slot, 21 bits per slot (a worker walks far fewer than 2^21 pages);
  // producer: slots whose last page was copied (bits)
  uint64_t slot_uses = 0;
  uint32_t slot_loaded = 0;
  const auto uses_of = [&](uint32_t sl) { return (uint32_t)(slot_uses >> (21 * sl)) & 0x1fffffu; };
  uint32_t g_sig = 0;                  // score signaler: pages signalled
  uint32_t s_use[2] = {0u, 0u};        // score MMA: times each score buffer was written
  uint32_t s_seen = 0;                 // softmax group: pages of this group processed
  uint32_t it_cnt = 0;                 // items (MMA issuers, softmax, value warps)
  // value producer: messages copied, low-part pages copied, items walked;
  // per probability unit and low-part buffer the item (+1) whose epilogue
  // stages in it (0: none), and per low-part buffer its last page
  uint32_t g_msg = 0, n_lo = 0, p_items = 0;
  uint32_t hi_epi[kHiUnits] = {0u, 0u, 0u};
  uint32_t lo_epi[kLoBufs] = {0u, 0u}, lo_occ[kLoBufs] = {0xffffffffu, 0xffffffffu};

  for (int offset = 0;; offset += kMaxItems) {
    plan_batch(a, w, offset, &ctl);
    const int n_items = ctl.n_batch;
    if (n_items == 0) break;

    if (warp == 0) {
      // ============================================================ producer
      // The whole warp walks the batch's pages in order; lane k holds the
      // block ids of pages 32c + k of the current chunk c and of the next one
      // (loaded a chunk ahead), lane 0 issues the copies: one per page.
      const int total = ctl.n_flat;
      // the score CTA's page copies stay in L2 for the value CTA's copy of the
      // same latents, which is their last use
      const uint64_t pol = rank == 0 ? policy_evict_last() : policy_evict_first();
      int cur = lane < total ? block_of(a, &ctl, n_items, lane) : -1;
      int nxt = 32 + lane < total ? block_of(a, &ctl, n_items, 32 + lane) : -1;
      if (rank == 0) {
        for (int f = 0; f < kPrefetch && f < total; ++f) {
          const int bp = __shfl_sync(0xffffffffu, cur, f);
          if (lane == 0 && bp >= 0 && bp < a.num_blocks) tma_prefetch_l2_4d(&tm_page, 0, 0, 0, bp * 8);
        }
      }
      int ip = 0;                          // item of page f
      for (int f = 0; f < total; ++f) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        while (ip + 1 < n_items && ctl.item_flat[ip + 1] <= f) ++ip;
        if ((f & 31) == 0 && f > 0) {
          cur = nxt;
          nxt = f + 32 + lane < total ? block_of(a, &ctl, n_items, f + 32 + lane) : -1;
        }
        const int pf = f + kPrefetch;
        const int bpf = __shfl_sync(0xffffffffu, (pf >> 5) == (f >> 5) ? cur : nxt, pf & 31);
        const int bk = __shfl_sync(0xffffffffu, cur, f & 31);
        if (lane == 0) {
          const bool ok = bk >= 0 && bk < a.num_blocks;
          // an invalid block is read past the pool's end: TMA fills zeros
          const int y = (ok ? bk : a.num_blocks) * 8;
          if (rank == 0) {
            if (!ok) atomicOr(a.err, kErrBadIndex);
            if (pf < total && bpf >= 0 && bpf < a.num_blocks) tma_prefetch_l2_4d(&tm_page, 0, 0, 0, bpf * 8);
            const int kp = f - ctl.item_flat[ip];   // page of its item
            const uint32_t sl = page_slot((kp & 1) ? g_unit - 1 : g_unit, kp & 1);
            if (!(kp & 1)) ++g_unit;
            slot_loaded &= ~(1u << sl);
            if (uses_of(sl) > 0 &&
                !mbar_wait(&ctl.slot_empty[sl], (uses_of(sl) - 1) & 1, abort_flag, wait_ns)) {
              fail(&ctl, a.err);
            } else if (!(a.skip_load > 0 && w == 0 && g_prod + 1 == (uint32_t)a.skip_load)) {
              mbar_arrive_expect_tx(&ctl.slot_full[sl], kPageBytes);
              tma_load_4d(smem + sl * kPageBytes, &tm_page, &ctl.slot_full[sl], 0, 0, 0, y, pol);
              g_issue = g_prod + 1;
              slot_loaded |= 1u << sl;
            }
            slot_uses += 1ull << (21 * sl);
          } else {
            const uint32_t g = g_prod, vs = g % kVSlots;
            bool ok2 = g < (uint32_t)kVSlots ||
                       mbar_wait(&ctl.v_empty[vs], ((g / kVSlots) - 1) & 1, abort_flag, wait_ns);
            if (ok2) {
              mbar_arrive_expect_tx(&ctl.v_full[vs], kVBytes);
              tma_load_4d(smem + kOffV + vs * kVBytes, &tm_v, &ctl.v_full[vs], 0, 0, 0, y, pol);
              tma_load_4d(smem + kOffV + vs * kVBytes + kVBytes / 2, &tm_v, &ctl.v_full[vs], 0, 0, 0, y + 4, pol);
              ++g_issue;
            }
            // page g's message: probabilities and row info into unit g % 3,
            // low parts (if any) into the next low-part buffer.  The unit was
            // last read by page g - 3's value MMAs; a unit or buffer that
            // held an item's last page is the staging area of its epilogue.
            const uint32_t gs = g % kGSlots, u = g % kHiUnits;
            const uint32_t K = p_items + (uint32_t)ip;
            const bool last_in_item = f + 1 == ctl.item_flat[ip + 1];
            if (ok2) ok2 = mbar_wait_cluster(&ctl.p_ready[gs], (g / kGSlots) & 1, abort_flag, wait_ns);
            if (ok2 && g >= (uint32_t)kHiUnits)
              ok2 = mbar_wait(&ctl.pv_done[(g - kHiUnits) & 7], ((g - kHiUnits) >> 3) & 1, abort_flag, wait_ns);
            if (ok2 && hi_epi[u]) ok2 = wait_count(&ctl.epi_count, hi_epi[u], abort_flag, wait_ns);
            const uint32_t fl = *reinterpret_cast<volatile uint32_t*>(&ctl.pflag_in[gs]);
            const bool lo = (fl & kFlagLo) != 0;
            const uint32_t lb = n_lo % kLoBufs;
            if (ok2 && lo) {
              // the buffer's last page: pages up to g - 3 are known to be done;
              // a more recent one is waited for here (the pv_done ring is
              // indexed by page, so an old page must not be waited for by parity)
              const uint32_t occ = lo_occ[lb];
              if (occ != 0xffffffffu && occ + kHiUnits > g)
                ok2 = mbar_wait(&ctl.pv_done[occ & 7], (occ >> 3) & 1, abort_flag, wait_ns);
              if (ok2 && lo_epi[lb]) ok2 = wait_count(&ctl.epi_count, lo_epi[lb], abort_flag, wait_ns);
            }
            if (!ok2) {
              fail(&ctl, a.err);
            } else {
              ctl.uflag[g & 7] = fl | (lb << 8);
              // the score CTA's writes of the message, acquired above, before
              // the bulk copies read them
              fence_proxy_async_global();
              const unsigned char* src = gmsg + (size_t)gs * kMsgBytes;
              mbar_arrive_expect_tx(&ctl.msg_full[u], kHiBytes + (lo ? kPBytes : 0));
              bulk_load_g2s(smem + kOffHi + u * kHiBytes, src, kHiBytes, &ctl.msg_full[u]);
              if (lo) bulk_load_g2s(smem + kOffLo + lb * kPBytes, src + kHiBytes, kPBytes, &ctl.msg_full[u]);
              hi_epi[u] = last_in_item ? K + 1 : 0u;
              if (lo) {
                lo_occ[lb] = g;
                lo_epi[lb] = last_in_item ? K + 1 : 0u;
                ++n_lo;
              }
              ++g_msg;
            }
          }
        }
        ++g_prod;
        __syncwarp();
      }
      p_items += (uint32_t)n_items;
    } else if (warp == 1) {
      // ============================================================ MMA issuer
      if (lane == 0) {
        if (rank == 0) {
          const uint32_t idS = idesc_bf16_f32(128, 64, 0, 0);
          const uint32_t idS2 = idesc_bf16_f32(128, 128, 0, 0);
          uint32_t g = g_page;
          for (int ii = 0; ii < n_items && !*abort_flag; ++ii) {
            const Item it = ctl.items[ii];
            const int n = it.j1 - it.j0;
            bool ok = mbar_wait(&ctl.q_ready, it_cnt & 1, abort_flag, wait_ns);
            // The item's pages in units (page_slot): a pair in slots (0, 1)
            // or (1, 2), scored as ONE operand of 128 tokens (the upper slot
            // continues the lower one's 9 KB stride), or an odd last page
            // alone.  The first page's scores always land at kTmemS; a pair in
            // (1, 2) holds its second page in the lower slot, so the operand
            // starts there and the scores start 64 columns lower.
            for (int k = 0; ok && k < n; k += 2) {
              const bool pair = k + 1 < n;
              const uint32_t sx = page_slot(g_unit, 0);
              ++g_unit;
              if (s_use[0] > 0) ok = mbar_wait(&ctl.s_free[0], (s_use[0] - 1) & 1, abort_flag, wait_ns);
              if (ok && pair && s_use[1] > 0) ok = mbar_wait(&ctl.s_free[1], (s_use[1] - 1) & 1, abort_flag, wait_ns);
              if (ok) ok = mbar_wait(&ctl.slot_full[sx], uses_of(sx) & 1, abort_flag, wait_ns);
              if (ok && pair) ok = mbar_wait(&ctl.slot_full[1], uses_of(1) & 1, abort_flag, wait_ns);
              if (!ok) break;
              tc_fence_after();
              // B = a page's tokens (K-major SW128, 8-token groups 9 KB
              // apart); chunk c starts 1 KB further, a K-step of 16 dims 32 B
              const uint32_t lo_slot = pair && sx == 2 ? 1u : sx;
              const uint64_t b0 = sdesc_sw128(smem_u32(smem + lo_slot * kPageBytes), 16, 9216);
              const uint32_t d = tmem + (pair && sx == 2 ? kTmemS - 64 : kTmemS);
              const uint32_t idN = pair ? idS2 : idS;
#pragma unroll 1
              for (int c = 0; c < 9; ++c)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ts(d, tmem + (uint32_t)(8 * (4 * c + kk)), b0 + (uint64_t)(64 * c + 2 * kk), idN,
                         (c | kk) ? 1u : 0u);
              mma_commit(&ctl.slot_empty[sx]);
              mma_commit(&ctl.s_full[0]);
              ++s_use[0];
              slot_uses += 1ull << (21 * sx);
              if (pair) {
                mma_commit(&ctl.slot_empty[1]);
                mma_commit(&ctl.s_full[1]);
                ++s_use[1];
                slot_uses += 1ull << 21;
              }
              g += pair ? 2 : 1;
            }
            if (!ok) { fail(&ctl, a.err); break; }
            mma_commit(&ctl.q_free);
            ++it_cnt;
          }
          g_page = g;
        } else {
          const uint32_t idPV = idesc_bf16_f32(128, 256, 0, 1);
          for (int ii = 0; ii < n_items && !*abort_flag; ++ii) {
            const Item it = ctl.items[ii];
            // the previous item's epilogue must have read O before it is overwritten
            bool ok = it_cnt == 0 || mbar_wait(&ctl.o_free, (it_cnt - 1) & 1, abort_flag, wait_ns);
            for (int i = 0; ok && i < it.j1 - it.j0; ++i) {
              const uint32_t g = g_page + i, vs = g % kVSlots;
              ok = mbar_wait(&ctl.vready[g & 7], (g >> 3) & 1, abort_flag, wait_ns);
              if (ok) ok = mbar_wait(&ctl.v_full[vs], (g / kVSlots) & 1, abort_flag, wait_ns);
              if (!ok) break;
              tc_fence_after();
              const uint32_t flags = *reinterpret_cast<const volatile uint32_t*>(&ctl.uflag[g & 7]);
              const bool lo = (flags & kFlagLo) != 0;
              // B = V (MN-major SW128): 64-dim chunks 1 KB apart along N,
              // 8-token groups 8 KB apart along K; a K-step is 16 tokens
              const uint64_t bv = sdesc_sw128(smem_u32(smem + kOffV + vs * kVBytes), 1024, 8192);
              // A = P chunk-major: 16-byte chunk c (tokens 8c .. 8c + 7) of row r at
              // c * 2048 + r * 16, the canonical K-major layout without swizzle
              // (core matrices 2 KB apart along K, 128 B apart along M); a K-step
              // of 16 tokens is two chunks, 4 KB
              const uint64_t ah = sdesc_noswz(smem_u32(smem + kOffHi + (g % kHiUnits) * kHiBytes), 2048, 128);
              const uint64_t al = sdesc_noswz(smem_u32(smem + kOffLo + ((flags >> 8) & 1u) * kPBytes), 2048, 128);
#pragma unroll
              for (int nh = 0; nh < 2; ++nh) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // 64 tokens, K-step 16
                  mma_ss(tmem + nh * 256, ah + (uint64_t)(256 * kk), bv + (uint64_t)(1024 * kk + 256 * nh), idPV,
                         (i > 0 || kk > 0) ? 1u : 0u);
                if (lo) {
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)   // the same V rows, A = low parts
                    mma_ss(tmem + nh * 256, al + (uint64_t)(256 * kk), bv + (uint64_t)(1024 * kk + 256 * nh), idPV, 1u);
                }
              }
              mma_commit(&ctl.v_empty[vs]);
              mma_commit(&ctl.pv_done[g & 7]);
            }
            if (!ok) { fail(&ctl, a.err); break; }
            g_page += it.j1 - it.j0;
            ++it_cnt;
          }
        }
      }
      __syncwarp();
    } else if (rank == 0 && warp <= 9) {
      // ============================================================ softmax (score CTA)
      // Two groups of four warps: warps 2-5 take the first page of each pair
      // of an item's pages (and an odd last page), warps 6-9 the second.
      // Warp w owns TMEM lane quarter w & 3 (rows 32 (w & 3) .. + 31), one
      // row per thread over all 64 tokens of a page.  Each page's reference
      // max follows from the previous page's (passed between the groups
      // through `mref`); a page's message carries the reference its
      // probabilities are relative to, and the value CTA rescales when
      // consecutive pages differ.
      const int grp = warp >= 6 ? 1 : 0;
      const int q4 = warp & 3;
      const int r = 32 * q4 + lane;
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
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
        // the previous item's scores, which read the query, are complete
        // (one phase of q_free per item; a group is never more than one item
        // ahead, because the scores of an item wait for its query)
        if (it_cnt > 0 && !warp_wait(&ctl.q_free, (it_cnt - 1) & 1, abort_flag, wait_ns)) { fail(&ctl, a.err); break; }
        load_query_row(a, it, rows, tmem, lane_off, r, grp, &ctl.q_ready);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int k = 0; k < n; ++k) {
          const uint32_t g = g_page + k, gs = g % kGSlots;
          if ((k & 1) != grp) continue;   // group 0 the first page of each pair, group 1 the second
          const int j = it.j0 + k;
          const bool last_page = k + 1 == n;
          const int bk = __ldg(a.block_table + (size_t)it.b * a.max_blocks + j);
          const bool page_ok = bk >= 0 && bk < a.num_blocks;
          if (!warp_wait(&ctl.s_full[grp], s_seen & 1, abort_flag, wait_ns)) { ok = false; break; }
          ++s_seen;
          tc_fence_after();
          float x[64];
          // the first page of unit u at kTmemS; the second 64 columns above,
          // or below when the pair sits in slots (1, 2)
          const uint32_t u = g_unit + (uint32_t)(k >> 1);
          const uint32_t scol = grp == 0 ? kTmemS : (page_slot(u, 0) == 2u ? kTmemS - 64 : kTmemS + 64);
          tmem_ld64(tmem + lane_off + scol, x);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.s_free[grp]);     // score buffer reusable
          // mask (tokens past the visible range, a bad block id, padding rows)
          const int tok0 = j * kPage;
          if (!page_ok || tok0 + 63 > L - a.T_q || r >= rows_g) {
            const int lim_page = page_ok ? lim : -1;
#pragma unroll
            for (int q = 0; q < 64; ++q) x[q] = (tok0 + q <= lim_page) ? x[q] : -INFINITY;
          }
          float mx = x[0];
#pragma unroll
          for (int q = 1; q < 64; ++q) mx = fmaxf(mx, x[q]);
          const float m_page = mx * sl2;
          // The page's reference max: the previous page's (sent by the other
          // group, which takes the item's other pages) unless this page's max
          // exceeds it by more than 2^8.  So the references of an item's pages
          // never decrease and the value CTA only ever scales O down.  The
          // references go through `mref`, tagged with page index + 1.
          float m_prev_ref = -INFINITY;
          volatile unsigned long long* mr = &ctl.mref[r];
          if (k > 0) {
            unsigned long long e = 0;
            if (!__all_sync(0xffffffffu, wait_tag(mr, g, &e, abort_flag, wait_ns))) { ok = false; break; }
            m_prev_ref = __uint_as_float((uint32_t)e);
          }
          const float m_new = m_page > m_prev_ref + kRescaleThreshold ? m_page : m_prev_ref;
          *mr = ((unsigned long long)(g + 1) << 32) | __float_as_uint(m_new);
          if (m_new != m_run) {
            l_run = m_run == -INFINITY ? 0.f : l_run * ex2(m_run - m_new);
            m_run = m_new;
          }
          // Precision of the bf16 probabilities: when a page's largest
          // probability is not small against this group's sum for the row so
          // far, the warp also sends the low bf16 parts (p - bf16(p)) of its
          // rows.  The item's last page always sends them: its buffers then
          // give the value CTA's epilogue its staging space.
          const bool lo = __any_sync(0xffffffffu, ex2(m_page - m_run) >= l_run) || last_page;
          // the page's message slot must have been read by the value CTA
          if (g >= (uint32_t)kGSlots &&
              !warp_wait_cluster(&ctl.gfree[gs], ((g / kGSlots) - 1) & 1, abort_flag, wait_ns)) { ok = false; break; }
          unsigned char* msg = gmsg + (size_t)gs * kMsgBytes;
          {
            // probabilities rounded to bf16 (and the residuals rounded again),
            // in the layout the value CTA's MMA reads (K-major, no swizzle,
            // chunk-major)
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t pk[4], pl[4];
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const float p0 = ex2(fmaf(x[8 * c + 2 * e2], sl2, neg_m));
                const float p1 = ex2(fmaf(x[8 * c + 2 * e2 + 1], sl2, neg_m));
                pk[e2] = pack_bf16x2(p0, p1);
                // the row sum counts the rounded values the value MMA multiplies
                const float h0 = __uint_as_float(lo_half_f(pk[e2])), h1 = __uint_as_float(hi_half_f(pk[e2]));
                ps0 += h0;
                ps1 += h1;
                if (lo) {
                  pl[e2] = pack_bf16x2(p0 - h0, p1 - h1);
                  ps0 += __uint_as_float(lo_half_f(pl[e2]));
                  ps1 += __uint_as_float(hi_half_f(pl[e2]));
                }
              }
              // chunk-major (chunk c of row r at c * 2048 + r * 16): each store
              // instruction of the warp writes 512 contiguous bytes.  (Rows of
              // 128 bytes, one 16-byte piece per lane and instruction, cost the
              // score SM ~20%: the MMA-issuing thread stalls behind them.)
              const int off = c * 2048 + r * 16;
              *reinterpret_cast<uint4*>(msg + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              if (lo) *reinterpret_cast<uint4*>(msg + kHiBytes + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            // row info: the reference max and the sum of this page's
            // (rounded) probabilities
            *reinterpret_cast<float2*>(msg + kPBytes + r * 8) = make_float2(m_run, ps0 + ps1);
            l_run += ps0 + ps1;
          }
          if (lane == 0 && lo) atomicOr(&ctl.pflags[g & 7], kFlagLo | (16u << q4));
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.written[g & 7]);
        }
        if (!ok) { fail(&ctl, a.err); break; }
        g_page += n;
        g_unit += (uint32_t)(n + 1) / 2;
        ++it_cnt;
      }
    } else if (rank == 0 && warp == 10) {
      // ============================================================ signaler (score CTA)
      // once a softmax group has written page g's message: its flags into
      // the value CTA's shared memory, then an arrival at cluster scope there,
      // which releases every write of the message (they happen before it
      // through the `written` barrier)
      if (lane == 0) {
        const uint32_t peer_pready = mapa(smem_u32(&ctl.p_ready[0]), 1);   // + 8 * slot
        const uint32_t peer_pflag = mapa(smem_u32(&ctl.pflag_in[0]), 1);   // + 4 * slot
        const int total = ctl.n_flat;
        for (int f = 0; f < total && !*abort_flag; ++f) {
          const uint32_t g = g_sig, gs = g % kGSlots;
          if (!mbar_wait(&ctl.written[g & 7], (g >> 3) & 1, abort_flag, wait_ns)) {
            fail(&ctl, a.err);
            break;
          }
          const uint32_t fl = *reinterpret_cast<volatile uint32_t*>(&ctl.pflags[g & 7]);
          ctl.pflags[g & 7] = 0u;              // ready for page g + 8
          st_cluster_u32(peer_pflag + 4 * gs, fl);
          mbar_arrive_remote(peer_pready + 8 * gs);
          ++g_sig;
        }
      }
      __syncwarp();
    } else if (rank == 1 && warp <= 9) {
      // ============================================================ value CTA warps
      // warps 2-5 ("row warps", one row per thread): once a page's message
      // is in shared memory, zero the low parts of the row quarters that sent
      // none, rescale O rows when the reference max changes, zero the V rows
      // of a last page past the sequence end, keep the row sums;
      // warps 2-9: the epilogue, warp w writing rows 32 (w & 3) .. + 31 and
      // output columns [256 * (w >= 6), + 256)
      const int q4 = warp & 3;
      const int ch = warp >= 6 ? 1 : 0;
      const bool row_warp = warp < 6;
      const int r = 32 * q4 + lane;
      const int tq = threadIdx.x - 64;             // 0..127 (row warps)
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const uint32_t peer_gfree = mapa(smem_u32(&ctl.gfree[0]), 0);   // + 8 * slot
      float l_row = 0.f, m_prev = -INFINITY;
      for (int ii = 0; ii < n_items; ++ii) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        const Item it = ctl.items[ii];
        const int L = a.seqlens[it.b];
        const int Pb = pages_of(L, a.T_q, cap);
        const int n = it.j1 - it.j0;
        bool ok = true;
        if (row_warp) {
          for (int i = 0; i < n; ++i) {
            const uint32_t g = g_page + i;
            const int j = it.j0 + i;
            const uint32_t u = g % kHiUnits;
            if (!(ok = warp_wait(&ctl.msg_full[u], (g / kHiUnits) & 1, abort_flag, wait_ns))) break;
            const uint32_t fl = *reinterpret_cast<const volatile uint32_t*>(&ctl.uflag[g & 7]);
            const uint32_t lb = (fl >> 8) & 1u;
            const float2 info = *reinterpret_cast<const float2*>(smem + kOffHi + u * kHiBytes + kPBytes + r * 8);
            if ((fl & kFlagLo) && !(fl & (16u << q4))) {
              // this row quarter sent no low parts: its rows of the buffer are zero
              uint4* lz = reinterpret_cast<uint4*>(smem + kOffLo + lb * kPBytes);   // chunk-major
#pragma unroll
              for (int c = 0; c < 8; ++c) lz[128 * c + r] = make_uint4(0u, 0u, 0u, 0u);
              fence_proxy_async_smem();    // the value MMA reads these bytes
            }
            __syncwarp();
            // the copies of the message slot have landed: the score CTA may reuse it
            if (q4 == 0 && lane == 0) mbar_arrive_remote_relaxed(peer_gfree + 8 * (g % kGSlots));
            const float m_j = info.x, srow = info.y;
            // rescale factor of this row: O and l hold pages < j relative to
            // m_prev; this page's probabilities are relative to m_j
            float alpha = 1.f;
            if (i == 0) {
              l_row = 0.f;
              m_prev = m_j;
            } else if (m_j != -INFINITY && m_j != m_prev) {
              alpha = m_prev == -INFINITY ? 0.f : ex2(m_prev - m_j);
              m_prev = m_j;
            }
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
              // O rows rescaled before this page's value MMA: O holds pages < j
              if (!(ok = warp_wait(&ctl.pv_done[(g - 1) & 7], ((g - 1) >> 3) & 1, abort_flag, wait_ns))) break;
              tc_fence_after();
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
            }
            l_row = l_row * alpha + srow;
            if (j == Pb - 1 && (L & (kPage - 1)) != 0) {
              // last page: zero the V rows past the sequence end (they may hold NaN)
              const uint32_t vs = g % kVSlots;
              if (!(ok = warp_wait(&ctl.v_full[vs], (g / kVSlots) & 1, abort_flag, wait_ns))) break;
              const int nv = L & (kPage - 1);
              const int pieces = (kPage - nv) * 8 * 8;      // 16-byte pieces: tokens x chunks x 8
              uint4* vp = reinterpret_cast<uint4*>(smem + kOffV + vs * kVBytes);
              for (int q = tq; q < pieces; q += kRows) {
                const int tk = nv + q / 64, rem = q & 63;     // token, (chunk, piece)
                const int cc = rem >> 3, pc = rem & 7;
                vp[((tk >> 3) * 8192 + cc * 1024 + (tk & 7) * 128) / 16 + pc] = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
            }
            if (i == n - 1) {
              // the item's last page: lse (natural log), the merge record, and
              // the row sum for the epilogue warps
              ctl.lrow[r] = l_row;
              const int rb = kRows * it.g;
              if (r < min(kRows, rows - rb)) {
                const float lse = l_row > 0.f ? (m_prev + __log2f(l_row)) * kLn2 : -INFINITY;
                if (it.flags & 1) { if (a.lse) a.lse[(size_t)it.b * rows + rb + r] = lse; }
                else a.ws_lse[(size_t)(it.vb + w) * a.SR + r] = lse;
                if (r == 0 && it.j0 == 0) a.meta[it.vb] = make_int2(it.w_first, it.w_last);
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.vready[g & 7]);
            if (i == n - 1) {
              // O is final once the last page's value MMAs are done; the
              // epilogue stages in this page's buffers
              if (!(ok = warp_wait(&ctl.pv_done[g & 7], (g >> 3) & 1, abort_flag, wait_ns))) break;
              if (lane == 0) {
                if (q4 == 2) ctl.epi_lo = lb;
                mbar_arrive(&ctl.epi_go);
              }
            }
          }
        }
        if (ok && !warp_wait(&ctl.epi_go, it_cnt & 1, abort_flag, wait_ns)) ok = false;
        if (!ok) { fail(&ctl, a.err); break; }
        // ---- epilogue: normalise and write the item's 128 x 512 output, staged
        // in the last page's probability unit and low-part buffer (the last
        // page always has low parts), each warp 32 rows x 16 columns at a time
        tc_fence_after();
        const uint32_t gl = g_page + n - 1;
        uint8_t* ps_last = smem + kOffHi + (gl % kHiUnits) * kHiBytes;
        uint8_t* ps_lo = smem + kOffLo + ctl.epi_lo * kPBytes;
        const float l_fin = ctl.lrow[r];
        const float inv = l_fin > 0.f ? 1.f / l_fin : 0.f;
        const bool whole = it.flags & 1;
        const int rb = kRows * it.g;                            // first row of the row group
        const int grp_rows = min(32, min(kRows, rows - rb) - 32 * q4);   // real rows of this warp's group
        float* out_base = (whole ? a.o + ((size_t)it.b * rows + rb) * a.d_c
                                 : a.ws_o + (size_t)(it.vb + w) * a.SR * a.d_c) + 256 * ch;
        if (grp_rows > 0) out_base += (size_t)(32 * q4) * a.d_c;
        const int wi = warp - 2;
        uint8_t* box = wi < 4 ? ps_last + wi * 4096 : ps_lo + (wi - 4) * 4096;   // this warp's 4 KB
        if (grp_rows == 32) {
          // whole 32-row group: 32 x 32 fp32 boxes staged (SW128) and written by TMA
          const CUtensorMap* tmo = whole ? &tm_o : &tm_ws;
          const int row0 = (whole ? it.b * rows + rb : (it.vb + w) * a.SR) + 32 * q4;
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
          if (lane == 0) bulk_wait_read0();         // staging free before it is reused
          __syncwarp();
        }
        float4* stg = reinterpret_cast<float4*>(box);   // 32 rows x 4 float4
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
        // the staging areas are reused by later pages: wait until every
        // epilogue warp is done with them, then let the producer copy into them
        if (!warp_wait(&ctl.epi_done, it_cnt & 1, abort_flag, wait_ns)) { fail(&ctl, a.err); break; }
        if (warp == 2 && lane == 0) *reinterpret_cast<volatile uint32_t*>(&ctl.epi_count) = it_cnt + 1;
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
  // ---- drain: all MMAs complete, all copies done, then free TMEM
  if (rank == 1 && warp >= 2 && warp <= 9 && lane == 0) bulk_wait0();   // output stores complete
  if (warp == 1 && lane == 0) {
    mma_commit(&ctl.mma_final);
    if (!mbar_wait(&ctl.mma_final, 0, &ctl.never, wait_ns)) atomicOr(a.err, kErrTimeout);
  }
  if (warp == 0 && lane == 0) {
    // the last copies issued into each ring slot have landed
    if (rank == 0) {
      // each slot's last page copy (a skipped load, test hook, was not issued)
      for (uint32_t sl = 0; sl < (uint32_t)kSlots; ++sl)
        if (((slot_loaded >> sl) & 1u) &&
            !mbar_wait(&ctl.slot_full[sl], (uses_of(sl) - 1) & 1, &ctl.never, wait_ns))
          atomicOr(a.err, kErrTimeout);
    } else {
      for (uint32_t k = 0; k < (uint32_t)kVSlots && k < g_issue; ++k) {
        const uint32_t g = g_issue - 1 - k;
        if (!mbar_wait(&ctl.v_full[g % kVSlots], (g / kVSlots) & 1, &ctl.never, wait_ns))
          atomicOr(a.err, kErrTimeout);
      }
      for (uint32_t k = 0; k < (uint32_t)kHiUnits && k < g_msg; ++k) {
        const uint32_t g = g_msg - 1 - k;
        if (!mbar_wait(&ctl.msg_full[g % kHiUnits], (g / kHiUnits) & 1, &ctl.never, wait_ns))
          atomicOr(a.err, kErrTimeout);
      }
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
std::once_flag g_encode_once;
TensorMapEncodeFn g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) e = cudaErrorNotSupported;
    if (e == cudaSuccess) g_encode = reinterpret_cast<TensorMapEncodeFn>(fn);
    g_encode_err = e;
  });
  return g_encode_err;
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

// The pool [num_blocks, 64, 576] bf16 seen as 4-D: (64 dims of a chunk,
// 8 tokens of a group, 9 chunks, num_blocks * 8 groups).  A box of `chunks`
// chunks starting at chunk c0 and 8 groups is one page (or its latent
// half), laid out [group][chunk][token][dim] in shared memory.
cudaError_t make_page_map(CUtensorMap* m, const void* pool, long long num_blocks, uint32_t chunks,
                          uint32_t groups = 8) {
  cuuint64_t dims[4] = {64, 8, 9, (cuuint64_t)num_blocks * 8};
  cuuint64_t strides[3] = {576 * 2, 64 * 2, 8 * 576 * 2};
  cuuint32_t box[4] = {64, 8, chunks, groups};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor maps of recent calls, per host thread: a decode step usually passes
// the same cache, output and workspace as the step before, and encoding the
// four maps is a noticeable part of a call's host time.
struct MapCacheEntry {
  uint64_t key[5];
  CUtensorMap map;
  bool used;
};
constexpr int kMapCache = 8;
thread_local MapCacheEntry t_maps[kMapCache];
thread_local int t_map_next = 0;

template <typename F>
cudaError_t cached_map(CUtensorMap* m, uint64_t k0, uint64_t k1, uint64_t k2, uint64_t k3, uint64_t k4, F encode) {
  const uint64_t key[5] = {k0, k1, k2, k3, k4};
  for (int i = 0; i < kMapCache; ++i) {
    const MapCacheEntry& c = t_maps[i];
    if (c.used && c.key[0] == key[0] && c.key[1] == key[1] && c.key[2] == key[2] && c.key[3] == key[3] &&
        c.key[4] == key[4]) {
      *m = c.map;
      return cudaSuccess;
    }
  }
  const cudaError_t e = encode(m);
  if (e == cudaSuccess) {
    MapCacheEntry& c = t_maps[t_map_next];
    t_map_next = (t_map_next + 1) % kMapCache;
    for (int i = 0; i < 5; ++i) c.key[i] = key[i];
    c.map = *m;
    c.used = true;
  }
  return e;
}

constexpr int kMaxDev = 64;
std::atomic<int> g_max_clusters[kMaxDev];
std::atomic<bool> g_attr_set[kMaxDev];

cudaError_t set_smem_attr(int dev) {
  if (dev >= 0 && dev < kMaxDev && g_attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) g_attr_set[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace

bool tc_supported(int dtype, int H, int T_q, int d_c, int d_r) {
  // query rows (heads x query tokens) in groups of up to 128; a short group is padded
  return dtype == BF16 && d_c == 512 && d_r == 64 && H * T_q >= 1;
}

int tc_item_cost(int rows) {
  // Fixed cost of one work item, in pages: the score CTA loads the item's
  // query rows into tensor memory before its first scores, and the value CTA
  // drains 128 x 512 fp32 of output before the next item may start.
  return 2 + (3 * rows + 64) / 128;
}

int tc_workers(int num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return num_sms / 2;
  int n = g_max_clusters[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (set_smem_attr(dev) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  g_max_clusters[dev].store(n, std::memory_order_release);
  return n;
}

cudaError_t tensor_map_encoder(TensorMapEncodeFn* fn) {
  const cudaError_t e = get_encode();
  if (e == cudaSuccess) *fn = g_encode;
  return e;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  if ((long long)a.num_blocks * 8 >= (1LL << 31)) return cudaErrorInvalidValue;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = set_smem_attr(dev);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_page, tm_v, tm_o, tm_ws;
  const uint64_t cache_p = reinterpret_cast<uintptr_t>(a.cache);
  e = cached_map(&tm_page, 1, cache_p, (uint64_t)a.num_blocks, 9, 0,
                 [&](CUtensorMap* m) { return make_page_map(m, a.cache, a.num_blocks, 9); });
  if (e != cudaSuccess) return e;
  e = cached_map(&tm_v, 1, cache_p, (uint64_t)a.num_blocks, 8, 4,   // the 512 latent dims of half a page
                 [&](CUtensorMap* m) { return make_page_map(m, a.cache, a.num_blocks, 8, 4); });
  if (e != cudaSuccess) return e;
  // outputs and split parts: [rows, 512] fp32, written in 32 x 32 boxes
  const uint64_t rows = (uint64_t)a.T_q * a.H;
  const uint64_t o_rows = (uint64_t)a.B * rows, ws_rows = ((uint64_t)a.B * a.G + a.W) * a.SR;
  e = cached_map(&tm_o, 2, reinterpret_cast<uintptr_t>(a.o), (uint64_t)a.d_c, o_rows, 0,
                 [&](CUtensorMap* m) { return make_map(m, a.o, (uint64_t)a.d_c, o_rows, 32, 32, true); });
  if (e != cudaSuccess) return e;
  e = cached_map(&tm_ws, 2, reinterpret_cast<uintptr_t>(a.ws_o), (uint64_t)a.d_c, ws_rows, 0,
                 [&](CUtensorMap* m) { return make_map(m, a.ws_o, (uint64_t)a.d_c, ws_rows, 32, 32, true); });
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
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel, a, tm_page, tm_v, tm_o, tm_ws);
}

}  // namespace mla
