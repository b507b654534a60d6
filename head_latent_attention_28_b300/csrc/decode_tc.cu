// Tensor-core MLA decode for sm_103a: 128 query rows (heads x query tokens)
// per sequence, cached rows of 512 latent + 64 rotary bfloat16 numbers.
//
// What it computes is the latent-space attention of the absorbed MLA path
// ("Attention, Part 2: MQA, GQA and MLA", the absorbed inference path: score =
// latent query . latent + rotary query . rotary key, scaled, causal mask,
// softmax, value sum over the latents; "How DeepSeek Rewrote the Transformer":
// the value is the first d_c numbers of the cached row).
//
// How (B300-specific).  One split worker is a cluster of two CTAs on two SMs:
//  * CTA 0, the score CTA, keeps the whole 128 x 576 latent query in tensor
//    memory (A operand), streams full 64-token pages with TMA and computes
//    S = Q . C^T (M=128 rows, N=64 tokens, K=576) with tcgen05.mma into one of
//    three TMEM score buffers.  Eight softmax warps (two per row, 32 tokens
//    each) run a base-2 online softmax with a lazy running max (the output is
//    rescaled only when a row max grows by more than 2^8; exact after the
//    final division), round the probabilities to bf16 and ship them, with the
//    per-row rescale factors, to the value CTA as one 17 KB bulk copy through
//    distributed shared memory.
//  * CTA 1, the value CTA, keeps the full 128 x 512 fp32 output in tensor
//    memory (all 512 columns), streams the 512 latent dims of the same pages
//    (the second read of a page is an L2 hit) and accumulates O += P . V with
//    tcgen05.mma (A = P from shared memory, B = V MN-major, N = 2 x 256).
//    Four warps apply row rescales, zero the rows of a last page past the
//    sequence end (0 x NaN would poison O), and write the normalised output.
// The data flow is one-way (score CTA -> value CTA), so the distributed-
// shared-memory latency is pipelined, never on a round trip.  Both CTAs carry
// 1024-1152 MMA cycles per page: the pair is balanced.
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
constexpr int kRows = 128;               // query rows per sequence handled here
constexpr int kBox = 8192;               // 64 tokens x 64 dims x bf16
constexpr int kSStageBytes = 9 * kBox;   // score CTA: full 576-dim page
constexpr int kVStageBytes = 8 * kBox;   // value CTA: 512 latent dims
constexpr int kStagesBytes = 2 * kSStageBytes;   // two stages (both roles fit)
constexpr int kPBytes = kRows * 64 * 2;  // bf16 probabilities of one page (K-major, SW128)
constexpr int kInfoBytes = 16 + kRows * 8;       // header + (alpha, l) per row
constexpr int kPMsgBytes = kPBytes + kInfoBytes; // one bulk copy per page
constexpr int kPSlotBytes = 34816;       // P + info + room for a second P (34 KB)
constexpr int kSmemBytes = kStagesBytes + 2 * kPSlotBytes + 1024;
constexpr int kMaxItems = 64;            // work items planned per batch
// TMEM columns
constexpr uint32_t kTmemQ = 192;         // score CTA: 288 columns = 576 bf16 query dims
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint64_t kWaitNs = 2000000000ull;

struct Item {
  int b, j0, j1;            // sequence, page range [j0, j1)
  int w_first, w_last;      // workers holding the sequence's first and last page
  int flags;                // bit 0: this worker holds the whole sequence
};

struct SmemCtl {
  // score CTA
  uint64_t stage_full[2], stage_empty[2];
  uint64_t s_full[3], s_free[3];
  uint64_t q_ready, pfree[2];
  // value CTA
  uint64_t v_full[2], v_empty[2];
  uint64_t p_recv[2], pv_done[2];
  uint64_t resc_done, vz_done;
  uint64_t o_free;          // the epilogue has read O: the next item may overwrite it
  // both
  uint64_t grp, mma_final;
  uint32_t tmem_base;
  int abort;
  int never;                // stays 0: abort flag for the final drain waits
  int n_batch, n_total;
  int scan[kThreads / 32];
  float rowx[2][kRows];     // score CTA: per-half row maxima
  float rowl[2][kRows];     // score CTA: per-half row sums (last page of an item)
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
// Same page partition as the CUDA-core kernel (see part_begin / part_worker_of).
__device__ void plan_batch(const DecodeArgs& a, int w, int offset, SmemCtl* ctl) {
  const int tid = threadIdx.x;
  const int cap = a.max_blocks * kPage;
  int mine = 0;
  for (int b = tid; b < a.B; b += kThreads) mine += pages_of(a.seqlens[b], a.T_q, cap);
  int total;
  cta_excl_scan(mine, ctl->scan, &total);
  const long long T = total;
  const int Wa = part_active(T, a.W);
  int n_total = 0, n_batch = 0;
  if (T > 0 && w < Wa) {
    const long long p0 = part_begin(T, Wa, w), p1 = part_begin(T, Wa, w + 1);
    long long base = 0;
    int count = 0;
    for (int c0 = 0; c0 < a.B && base < p1; c0 += kThreads) {
      const int b = c0 + tid;
      const int P = b < a.B ? pages_of(a.seqlens[b], a.T_q, cap) : 0;
      int chunk_total;
      const int excl = cta_excl_scan(P, ctl->scan, &chunk_total);
      const long long S = base + excl;
      const int hit = (P > 0 && S < p1 && S + P > p0) ? 1 : 0;
      int hits;
      const int idx = count + cta_excl_scan(hit, ctl->scan, &hits);
      if (hit && idx >= offset && idx < offset + kMaxItems) {
        const long long g0 = S > p0 ? S : p0;
        const long long g1 = (S + P) < p1 ? (S + P) : p1;
        Item it;
        it.b = b;
        it.j0 = (int)(g0 - S);
        it.j1 = (int)(g1 - S);
        it.w_first = part_worker_of(T, Wa, S);
        it.w_last = part_worker_of(T, Wa, S + P - 1);
        it.flags = (it.j0 == 0 && it.j1 == P) ? 1 : 0;
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
decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tm_pool) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;                          // 2 page stages
  uint8_t* pslots = smem + kStagesBytes;           // 2 probability slots

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();         // 0: score CTA, 1: value CTA
  const int w = (int)cluster_id_x();
  volatile int* abort_flag = &ctl.abort;

  if (threadIdx.x == 0) {
    ctl.abort = 0;
    ctl.never = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.stage_full[i], 1);
      mbar_init(&ctl.stage_empty[i], 1);
      mbar_init(&ctl.pfree[i], 1);
      mbar_init(&ctl.v_full[i], 1);
      mbar_init(&ctl.v_empty[i], 1);
      mbar_init(&ctl.p_recv[i], 1);
      mbar_init(&ctl.pv_done[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.s_free[i], 8);
    }
    mbar_init(&ctl.q_ready, 8);
    mbar_init(&ctl.resc_done, 4);
    mbar_init(&ctl.vz_done, 4);
    mbar_init(&ctl.o_free, 4);
    mbar_init(&ctl.grp, rank == 0 ? 8 : 4);
    mbar_init(&ctl.mma_final, 1);
    if (rank == 1) {   // the first two pages' probabilities will arrive
      mbar_arrive_expect_tx(&ctl.p_recv[0], kPMsgBytes);
      mbar_arrive_expect_tx(&ctl.p_recv[1], kPMsgBytes);
    }
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
  const int rows = a.T_q * a.H;   // == kRows
  const int cap = a.max_blocks * kPage;

  uint32_t g_prod = 0, g_issue = 0, g_mma = 0, g_sm = 0;   // page counters per role
  uint32_t it_mma = 0;                                     // items (score MMA)
  uint32_t grp_phase = 0, n_resc = 0, n_vz = 0;

  for (int offset = 0;; offset += kMaxItems) {
    plan_batch(a, w, offset, &ctl);
    const int n_items = ctl.n_batch;
    if (n_items == 0) break;

    if (warp == 0) {
      // ============================================================ producer
      // (the whole warp walks the loop; lane 0 issues barriers and copies)
      const uint64_t pol = policy_evict_first();
      const int nbox = rank == 0 ? 9 : 8;
      const int stage_bytes = rank == 0 ? kSStageBytes : kVStageBytes;
      uint64_t* full = rank == 0 ? ctl.stage_full : ctl.v_full;
      uint64_t* empty = rank == 0 ? ctl.stage_empty : ctl.v_empty;
      for (int ii = 0; ii < n_items; ++ii) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const Item it = ctl.items[ii];
        for (int jb = it.j0; jb < it.j1; jb += 32) {
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
          const int jj = jb + lane;
          int blk = -1;
          if (jj < it.j1) blk = a.block_table[(size_t)it.b * a.max_blocks + jj];
          const int nj = min(32, it.j1 - jb);
          for (int k = 0; k < nj; ++k) {
            const int bk = __shfl_sync(0xffffffffu, blk, k);
            if (lane == 0 && !*abort_flag) {
              const uint32_t st = g_prod & 1;
              bool ok = true;
              if (g_prod >= 2) ok = mbar_wait(&empty[st], ((g_prod >> 1) - 1) & 1, abort_flag, kWaitNs);
              if (!ok) fail(&ctl, a.err);
              else {
                const bool valid = bk >= 0 && bk < a.num_blocks;
                if (!valid && rank == 0) atomicOr(a.err, kErrBadIndex);
                // an invalid block is read past the pool's end: TMA fills zeros
                const int y = valid ? bk * kPage : a.num_blocks * kPage;
                uint8_t* dst = stages + st * kSStageBytes;
                mbar_arrive_expect_tx(&full[st], stage_bytes);
                for (int bx = 0; bx < nbox; ++bx)
                  tma_load_2d(dst + bx * kBox, &tm_pool, &full[st], 64 * bx, y, pol);
                ++g_issue;
              }
            }
            ++g_prod;
            __syncwarp();
          }
        }
      }
    } else if (warp == 1) {
      // ============================================================ MMA issuer
      if (lane == 0) {
        if (rank == 0) {
          const uint32_t idS = idesc_bf16_f32(128, 64, 0, 0);
          for (int ii = 0; ii < n_items && !*abort_flag; ++ii) {
            const Item it = ctl.items[ii];
            bool ok = mbar_wait(&ctl.q_ready, it_mma & 1, abort_flag, kWaitNs);
            for (int i = 0; ok && i < it.j1 - it.j0; ++i) {
              const uint32_t g = g_mma + i, sb = g % 3;
              if (g >= 3) ok = mbar_wait(&ctl.s_free[sb], ((g / 3) - 1) & 1, abort_flag, kWaitNs);
              if (ok) ok = mbar_wait(&ctl.stage_full[g & 1], (g >> 1) & 1, abort_flag, kWaitNs);
              if (!ok) break;
              tc_fence_after();
              const uint8_t* st = stages + (g & 1) * kSStageBytes;
              for (int kk = 0; kk < 36; ++kk) {   // K = 576: query in TMEM, page in smem
                const uint64_t bd =
                    sdesc_sw128(smem_u32(st + (kk >> 2) * kBox + (kk & 3) * 32), 16, 1024);
                mma_ts(tmem + sb * 64, tmem + kTmemQ + kk * 8, bd, idS, kk > 0);
              }
              mma_commit(&ctl.s_full[sb]);
              mma_commit(&ctl.stage_empty[g & 1]);
            }
            if (!ok) { fail(&ctl, a.err); break; }
            g_mma += it.j1 - it.j0;
            ++it_mma;
          }
        } else {
          const uint32_t idPV = idesc_bf16_f32(128, 256, 0, 1);
          for (int ii = 0; ii < n_items && !*abort_flag; ++ii) {
            const Item it = ctl.items[ii];
            const int L = a.seqlens[it.b];
            const int Pb = pages_of(L, a.T_q, cap);
            // the previous item's epilogue must have read O before it is overwritten
            bool ok = it_mma == 0 || mbar_wait(&ctl.o_free, (it_mma - 1) & 1, abort_flag, kWaitNs);
            for (int i = 0; ok && i < it.j1 - it.j0; ++i) {
              const uint32_t g = g_mma + i, slot = g & 1;
              const int j = it.j0 + i;
              ok = mbar_wait(&ctl.p_recv[slot], (g >> 1) & 1, abort_flag, kWaitNs);
              if (!ok) break;
              const uint8_t* ps = pslots + slot * kPSlotBytes;
              const uint32_t flags = *reinterpret_cast<const volatile uint32_t*>(ps + kPBytes);
              if ((flags & 1u) && i > 0) {          // rows rescaled by the value warps
                ok = mbar_wait(&ctl.resc_done, n_resc & 1, abort_flag, kWaitNs);
                ++n_resc;
              }
              if (ok && j == Pb - 1 && (L & (kPage - 1)) != 0) {   // tail rows zeroed
                ok = mbar_wait(&ctl.vz_done, n_vz & 1, abort_flag, kWaitNs);
                ++n_vz;
              }
              if (ok) ok = mbar_wait(&ctl.v_full[g & 1], (g >> 1) & 1, abort_flag, kWaitNs);
              if (!ok) break;
              tc_fence_after();
              const uint8_t* vs = stages + (g & 1) * kSStageBytes;
              for (int nh = 0; nh < 2; ++nh) {
                for (int kk = 0; kk < 4; ++kk) {   // 64 tokens, K-step 16
                  const uint64_t ad = sdesc_sw128(smem_u32(ps + kk * 32), 16, 1024);
                  const uint64_t bd = sdesc_sw128(smem_u32(vs + nh * 4 * kBox + kk * 2048), kBox, 1024);
                  mma_ss(tmem + nh * 256, ad, bd, idPV, (i > 0 || kk > 0) ? 1 : 0);
                }
              }
              mma_commit(&ctl.v_empty[g & 1]);
              mma_commit(&ctl.pv_done[slot]);
            }
            if (!ok) { fail(&ctl, a.err); break; }
            g_mma += it.j1 - it.j0;
            ++it_mma;
          }
        }
      }
      __syncwarp();
    } else if (rank == 0) {
      // ============================================================ softmax (score CTA)
      const int q4 = warp & 3;
      const int half = warp >= 6 ? 1 : 0;          // tokens [32*half, 32*half + 32)
      const int r = 32 * q4 + lane;
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const uint32_t peer_pslots = mapa(smem_u32(pslots), 1);
      const uint32_t peer_precv0 = mapa(smem_u32(&ctl.p_recv[0]), 1);
      const uint32_t peer_precv1 = mapa(smem_u32(&ctl.p_recv[1]), 1);
      const int t = r / a.H;
      for (int ii = 0; ii < n_items; ++ii) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        const Item it = ctl.items[ii];
        const int L = a.seqlens[it.b];
        const int lim = a.causal ? (L - a.T_q + t) : (L - 1);
        const int n = it.j1 - it.j0;
        // the whole latent query row -> TMEM (A operand of the score MMA);
        // half 0 writes dims [0, 320), half 1 dims [320, 576)
        {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(a.q) + ((size_t)it.b * rows + r) * a.D) + half * 40;
          const int nchunk = half ? 4 : 5;
          for (int c = 0; c < nchunk; ++c) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 x = __ldg(src + c * 8 + u);
              v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
            }
            tmem_st32(tmem + lane_off + kTmemQ + half * 160 + 32 * c, v);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.q_ready);
        }
        float m_run = -INFINITY, l_half = 0.f;
        bool ok = true;
        for (int i = 0; i < n; ++i) {
          const uint32_t g = g_sm + i, sb = g % 3, slot = g & 1;
          const int j = it.j0 + i;
          const bool last = (i == n - 1);
          const int bk = __ldg(a.block_table + (size_t)it.b * a.max_blocks + j);
          const bool page_ok = bk >= 0 && bk < a.num_blocks;
          if (!warp_wait(&ctl.s_full[sb], (g / 3) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          float x[32];
          tmem_ld32(tmem + lane_off + sb * 64 + 32 * half, x);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.s_free[sb]);     // score buffer reusable
          // mask (tokens past the visible range, or a page with a bad block id)
          const int tok0 = j * kPage + 32 * half;
          if (!page_ok || tok0 + 31 > L - a.T_q) {
            const int lim_page = page_ok ? lim : -1;
#pragma unroll
            for (int k = 0; k < 32; ++k) x[k] = (tok0 + k <= lim_page) ? x[k] : -INFINITY;
          }
          float mx = x[0];
#pragma unroll
          for (int k = 1; k < 32; ++k) mx = fmaxf(mx, x[k]);
          ctl.rowx[half][r] = mx;
          uint8_t* ps = pslots + slot * kPSlotBytes;          // our staging for this page
          if (threadIdx.x == 64) {
            bool fr = true;
            if (g >= 2) fr = mbar_wait_cluster(&ctl.pfree[slot], ((g >> 1) - 1) & 1, abort_flag, kWaitNs);
            if (!fr) fail(&ctl, a.err);
            *reinterpret_cast<uint32_t*>(ps + kPBytes) = 0u;   // header flags
          }
          if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }   // [A]
          const float mo = ctl.rowx[half ^ 1][r];
          const float m_page = fmaxf(mx, mo) * sl2;
          const float m_new = fmaxf(m_run, m_page);
          const bool need = m_new > m_run + kRescaleThreshold;
          float alpha = 1.f;
          if (need) {
            alpha = ex2(m_run - m_new);     // 0 when m_run = -inf
            m_run = m_new;
            l_half *= alpha;
          }
          // probabilities, rounded to bf16 once; l sums the rounded values
          uint32_t pk[16];
          float psum = 0.f;
          const float neg_m = -m_run;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float p0 = x[2 * k] == -INFINITY ? 0.f : ex2(fmaf(x[2 * k], sl2, neg_m));
            const float p1 = x[2 * k + 1] == -INFINITY ? 0.f : ex2(fmaf(x[2 * k + 1], sl2, neg_m));
            pk[k] = pack_bf16x2(p0, p1);
            psum += __uint_as_float(lo_half_f(pk[k])) + __uint_as_float(hi_half_f(pk[k]));
          }
          l_half += psum;
          {
            uint4* prow = reinterpret_cast<uint4*>(ps + r * 128);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              prow[(4 * half + c) ^ (r & 7)] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
          float* info = reinterpret_cast<float*>(ps + kPBytes + 16);
          if (half == 0) info[2 * r] = alpha;
          if (__any_sync(0xffffffffu, need) && i > 0 && lane == 0)
            atomicOr(reinterpret_cast<uint32_t*>(ps + kPBytes), 1u);
          if (last) {
            ctl.rowl[half][r] = l_half;
            if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }
            const float l_tot = ctl.rowl[0][r] + ctl.rowl[1][r];
            if (half == 0) {
              info[2 * r + 1] = l_tot;
              const float lse = l_tot > 0.f ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
              const int wslot = it.b + w;
              if (it.flags & 1) { if (a.lse) a.lse[(size_t)it.b * rows + r] = lse; }
              else a.ws_lse[(size_t)wslot * rows + r] = lse;
              if (r == 0 && it.j0 == 0) a.meta[it.b] = make_int2(it.w_first, it.w_last);
            }
          }
          fence_proxy_async_smem();
          if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }   // [B]
          if (threadIdx.x == 64 && !*abort_flag)
            bulk_copy_to_peer(peer_pslots + slot * kPSlotBytes, ps, kPMsgBytes,
                              slot ? peer_precv1 : peer_precv0);
        }
        if (!ok) { fail(&ctl, a.err); break; }
        g_sm += n;
      }
    } else if (warp < 6) {
      // ============================================================ value CTA rows
      const int q4 = warp & 3;
      const int r = 32 * q4 + lane;
      const int tq = threadIdx.x - 64;             // 0..127
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const uint32_t peer_pfree0 = mapa(smem_u32(&ctl.pfree[0]), 0);
      const uint32_t peer_pfree1 = mapa(smem_u32(&ctl.pfree[1]), 0);
      for (int ii = 0; ii < n_items; ++ii) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        const Item it = ctl.items[ii];
        const int L = a.seqlens[it.b];
        const int Pb = pages_of(L, a.T_q, cap);
        const int n = it.j1 - it.j0;
        bool ok = true;
        float l_row = 0.f;
        for (int i = 0; i < n; ++i) {
          const uint32_t g = g_sm + i, slot = g & 1;
          const int j = it.j0 + i;
          uint8_t* ps = pslots + slot * kPSlotBytes;
          if (!warp_wait(&ctl.p_recv[slot], (g >> 1) & 1, abort_flag)) { ok = false; break; }
          const uint32_t flags = *reinterpret_cast<const volatile uint32_t*>(ps + kPBytes);
          const float* info = reinterpret_cast<const float*>(ps + kPBytes + 16);
          if (j == Pb - 1 && (L & (kPage - 1)) != 0) {
            // last page: zero the V rows past the sequence end (they may hold NaN)
            if (!warp_wait(&ctl.v_full[g & 1], (g >> 1) & 1, abort_flag)) { ok = false; break; }
            const int nv = L & (kPage - 1);
            uint4* vs = reinterpret_cast<uint4*>(stages + (g & 1) * kSStageBytes);
            const int per_box = (kPage - nv) * 8;
            for (int q = tq; q < 8 * per_box; q += kRows) {
              const int bx = q / per_box, rem = q - bx * per_box;
              vs[(bx * kBox + (nv + rem / 8) * 128) / 16 + (rem & 7)] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.vz_done);
          }
          if ((flags & 1u) && i > 0) {
            // rescale O rows before this page's value MMA: O holds pages < j
            if (!warp_wait(&ctl.pv_done[slot ^ 1], ((g - 1) >> 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const float alpha = info[2 * r];
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float o[64];
              tmem_ld64(tmem + lane_off + 64 * c, o);
              tmem_ld_wait();
              uint32_t u0[32], u1[32];
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                u0[k] = __float_as_uint(o[k] * alpha);
                u1[k] = __float_as_uint(o[32 + k] * alpha);
              }
              tmem_st32(tmem + lane_off + 64 * c, u0);
              tmem_st32(tmem + lane_off + 64 * c + 32, u1);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.resc_done);
          }
          if (i == n - 1) l_row = info[2 * r + 1];
          // this page's value MMA done: the slot may be refilled (the last
          // page's slot is released after the epilogue, which reuses it)
          if (!warp_wait(&ctl.pv_done[slot], (g >> 1) & 1, abort_flag)) { ok = false; break; }
          if (i < n - 1 && threadIdx.x == 64) {
            mbar_arrive_expect_tx(&ctl.p_recv[slot], kPMsgBytes);
            mbar_arrive_remote(slot ? peer_pfree1 : peer_pfree0);
          }
        }
        if (!ok) { fail(&ctl, a.err); break; }
        const uint32_t g_last = g_sm + n - 1, slot = g_last & 1;
        g_sm += n;
        // ---- epilogue: normalise and write the item's 128 x 512 output,
        // staged through the last page's slot for coalesced row writes
        tc_fence_after();
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        const bool whole = it.flags & 1;
        float* out_base = whole ? a.o + (size_t)it.b * rows * a.d_c
                                : a.ws_o + (size_t)(it.b + w) * rows * a.d_c;
        float4* stage_o = reinterpret_cast<float4*>(pslots + slot * kPSlotBytes);
        if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { fail(&ctl, a.err); break; }  // l read
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float o[64];
          tmem_ld64(tmem + lane_off + 64 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k)
            stage_o[r * 16 + (k ^ (r & 7))] =
                make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv, o[4 * k + 3] * inv);
          if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }
#pragma unroll 4
          for (int idx = tq; idx < kRows * 16; idx += kRows) {
            const int row = idx >> 4, c16 = idx & 15;
            reinterpret_cast<float4*>(out_base + (size_t)row * a.d_c + 64 * c)[c16] =
                stage_o[row * 16 + (c16 ^ (row & 7))];
          }
          if (!group_sync(&ctl.grp, grp_phase, abort_flag)) { ok = false; break; }
        }
        if (!ok) { fail(&ctl, a.err); break; }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.o_free);      // O may be overwritten now
        if (threadIdx.x == 64) {
          mbar_arrive_expect_tx(&ctl.p_recv[slot], kPMsgBytes);
          mbar_arrive_remote(slot ? peer_pfree1 : peer_pfree0);
        }
      }
    }
    __syncthreads();
    if (*abort_flag) break;
    if (offset + kMaxItems >= ctl.n_total) break;
  }

  // ---- drain: all MMAs complete, all TMA loads landed, then free TMEM
  if (warp == 1 && lane == 0) {
    mma_commit(&ctl.mma_final);
    if (!mbar_wait(&ctl.mma_final, 0, &ctl.never, kWaitNs)) atomicOr(a.err, kErrTimeout);
  }
  if (warp == 0 && lane == 0) {
    uint64_t* full = rank == 0 ? ctl.stage_full : ctl.v_full;
    for (uint32_t k = 0; k < 2u && k < g_issue; ++k) {
      const uint32_t g = g_issue - 1 - k;
      if (!mbar_wait(&full[g & 1], (g >> 1) & 1, &ctl.never, kWaitNs)) atomicOr(a.err, kErrTimeout);
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
                     uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int g_max_clusters[64] = {};

}  // namespace

bool tc_supported(int dtype, int H, int T_q, int d_c, int d_r) {
  return dtype == BF16 && d_c == 512 && d_r == 64 && H * T_q == kRows;
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

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  if ((long long)a.num_blocks * kPage >= (1LL << 31)) return cudaErrorInvalidValue;
  CUtensorMap tm_pool;
  e = make_map(&tm_pool, a.cache, (uint64_t)a.D, (uint64_t)a.num_blocks * kPage, 64, 64);
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
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel, a, tm_pool);
}

}  // namespace mla
