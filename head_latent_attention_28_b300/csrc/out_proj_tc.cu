// The output projections of the absorbed path on the tensor cores, bf16
// weights ("Attention, Part 2: MQA, GQA and MLA" and "How DeepSeek Rewrote
// the Transformer", the absorbed inference path: the value up-projection
// W^UV_h is applied once to the attended latent o_lat, then W^O; or W^UV is
// folded into W^O, so o_lat goes through one matrix per head).
//
//   unmerged  o[n, h*d_h + v] = sum_c W^UV[h*d_h + v, c] * o_lat[n, h, c]
//             out[n, j]       = sum_k W^O[j, k] * o[n, k]
//   merged    W_m[j, h*d_c + c] = sum_v W^O[j, h*d_h + v] * W^UV[h*d_h + v, c]
//             out[n, j]         = sum_{h, c} W_m[j, h*d_c + c] * o_lat[n, h, c]
//
// All are C = A . B^T contractions with A and B K-major bf16 in global
// memory, done by one kernel (gemm_tn_kernel): TMA copies 128 x 64 tiles of
// A and 256 x 64 tiles of B into a ring of stages (128-byte swizzle), one
// thread issues tcgen05.mma (M = 128, N = 256, K = 16) into a 128 x 256 fp32
// accumulator in tensor memory, and four warps drain it.  In the unmerged
// path the fp32 activations (o_lat, then o) enter as two bf16 matrices, the
// rounded value and the rounded remainder (hi + lo, 16 significant bits),
// multiplied by the same weight tile: the products keep about fp32 accuracy
// at twice the MMAs, which the weight stream hides at decode batch sizes.
//  * The first unmerged projection is batched over heads (CTA z = h: o_lat's
//    column block h times W^UV_h), the second splits K = H * d_h across the
//    grid like the merged output below.
//  * The merge (once per set of weights) is batched over heads: CTA z = h
//    multiplies W^O's column block h (rows of A) by W^UV_h, handed in
//    transposed ([d_c, d_h] per head, a small copy made first), and writes
//    its tile of W_m rounded to bf16.
//  * The merged output splits K = H * d_c across the grid (split-K): o_lat
//    is rounded to bf16 first (the merged weights are bf16 too), each CTA
//    writes fp32 partial sums of its K range, and a last kernel adds the
//    partials in a fixed order (deterministic).
// At decode batch sizes the merged output is bound by reading W_m
// (d * H * d_c bf16), which is larger than W^UV and W^O together whenever
// d_h < d_c; the unmerged pair of projections (mla_absorb_output) reads less.
//
// Every wait is bounded (2 s); on expiry the kernel records MLA_ERR_TIMEOUT,
// lets its copies land, frees tensor memory and writes nothing.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int kGT = 128;                    // threads (warp 0 copies, warp 1 issues MMAs, all drain)
constexpr int kGM = 128;                    // C rows per CTA (tensor-memory lanes)
constexpr int kGN = 256;                    // C columns per CTA (tensor-memory columns)
constexpr int kGK = 64;                     // K per stage: one 128-byte swizzle row of bf16
constexpr int kGABytes = kGM * kGK * 2;     // 16 KB
constexpr int kGBBytes = kGN * kGK * 2;     // 32 KB
constexpr uint64_t kGWaitNs = 2000000000ull;
// A as one bf16 matrix: stages [A 16 KB][B 32 KB] x 4; as hi + lo: [A hi][A lo][B] x 3
template <bool kSplitA> struct GemmShape {
  static constexpr int kABytes = kSplitA ? 2 * kGABytes : kGABytes;
  static constexpr int kStageBytes = kABytes + kGBBytes;
  static constexpr int kStages = kSplitA ? 3 : 4;
  static constexpr int kSmem = kStages * kStageBytes + 1024;
};
// C: fp32 partial sums (split-K), bf16, or bf16 rounded value + remainder
enum { kOutF32Part = 0, kOutBf16 = 1, kOutBf16HiLo = 2 };

struct GemmArgs {
  int M, N;        // C rows < M and columns < N are written (columns per z in batched mode)
  int K;           // contraction length (per z in batched mode)
  int k_split;     // split mode: K per CTA along z (a multiple of 64)
  int a_kz;        // batched mode: A's K offset per z
  int b_nz;        // batched mode: B's row offset per z
  float* c32;      // split mode: partial sums [z][M][ldc]
  __nv_bfloat16* c16;   // batched mode: C [M][ldc], columns from z * c_nz
  __nv_bfloat16* c16lo; // batched hi/lo mode: the remainders, same layout
  int ldc, c_nz;
  unsigned* err;
};

// 32 consecutive numbers rounded to bf16 (the first `valid` of them stored)
__device__ __forceinline__ void store_bf16_32(__nv_bfloat16* dst, const float (&v)[32], int valid) {
  if (valid >= 32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t*>(&p);
      }
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid) dst[i] = __float2bfloat16_rn(v[i]);
  }
}

template <bool kBatched, bool kSplitA, int kOut>
__global__ void __launch_bounds__(kGT, 1)
gemm_tn_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tm_a,
               const __grid_constant__ CUtensorMap tm_alo, const __grid_constant__ CUtensorMap tm_b) {
  using Sh = GemmShape<kSplitA>;
  constexpr int kGStages = Sh::kStages, kGStageBytes = Sh::kStageBytes, kAB = Sh::kABytes;
  extern __shared__ uint8_t gm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gm_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t full[kGStages], empty[kGStages], done;
  __shared__ uint32_t tbase;
  __shared__ int failed, never;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kGN, m0 = blockIdx.y * kGM, z = blockIdx.z;
  const int k_lo = kBatched ? 0 : z * a.k_split;
  const int k_hi = kBatched ? a.K : min(a.K, k_lo + a.k_split);
  const int nk = (k_hi - k_lo + kGK - 1) / kGK;         // >= 1 (the launcher sees to it)
  const int a_k0 = kBatched ? z * a.a_kz : 0;
  const int b_r0 = (kBatched ? z * a.b_nz : 0) + n0;
  if (threadIdx.x == 0) {
    failed = 0;
    never = 0;
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 0) tmem_alloc(&tbase, kGN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;

  if (warp == 0 && lane == 0) {
    // ---- copies: stage kb % 4 holds A[m0.., k] and B[n0.., k] for k = k_lo + 64 kb
    const uint64_t pol_a = policy_evict_last();    // A is re-read by the CTAs of other columns
    const uint64_t pol_b = policy_evict_first();   // B is read once
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kGStages;
      if (kb >= kGStages && !mbar_wait(&empty[s], ((kb / kGStages) - 1) & 1, &failed, kGWaitNs)) {
        failed = 1;
        atomicOr(a.err, kErrTimeout);
        break;
      }
      uint8_t* sa = smem + s * kGStageBytes;
      mbar_arrive_expect_tx(&full[s], kGStageBytes);
      tma_load_2d(sa, &tm_a, &full[s], a_k0 + k_lo + kGK * kb, m0, pol_a);
      if (kSplitA) tma_load_2d(sa + kGABytes, &tm_alo, &full[s], a_k0 + k_lo + kGK * kb, m0, pol_a);
      tma_load_2d(sa + kAB, &tm_b, &full[s], k_lo + kGK * kb, b_r0, pol_b);
      issued = kb + 1;
    }
    // the copies in flight land before the CTA exits
    for (int kb = issued - 1; kb >= 0 && kb >= issued - kGStages; --kb)
      if (!mbar_wait(&full[kb % kGStages], (kb / kGStages) & 1, &never, kGWaitNs)) atomicOr(a.err, kErrTimeout);
  } else if (warp == 1 && lane == 0) {
    // ---- MMAs: 128 x 256 += (128 x 64) . (256 x 64)^T per stage, four K-steps of 16
    const uint32_t id = idesc_bf16_f32(kGM, kGN, 0, 0);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kGStages;
      if (!mbar_wait(&full[s], (kb / kGStages) & 1, &failed, kGWaitNs)) { ok = false; break; }
      tc_fence_after();
      const uint8_t* sa = smem + s * kGStageBytes;
      const uint64_t ad = sdesc_sw128(smem_u32(sa), 16, 1024);
      const uint64_t bd = sdesc_sw128(smem_u32(sa + kAB), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_ss(tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), id, (kb | kk) ? 1u : 0u);
        if (kSplitA)   // the remainders: + 16 KB is + 1024 in descriptor units
          mma_ss(tmem, ad + (uint64_t)(1024 + 2 * kk), bd + (uint64_t)(2 * kk), id, 1u);
      }
      mma_commit(&empty[s]);
    }
    if (!ok) {
      failed = 1;
      atomicOr(a.err, kErrTimeout);
    }
    mma_commit(&done);   // also tracks the MMAs already issued when a wait gave up
  }
  __syncwarp();

  // ---- drain: warp w holds C rows m0 + 32 w .. + 31 (one per lane)
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&done, 0, &never, kGWaitNs)) && !failed;
  tc_fence_after();
  const int r = m0 + 32 * warp + lane;
  if (ok) {
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
#pragma unroll 1
    for (int c = 0; c < kGN / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_off + 32 * c, v);
      tmem_ld_wait();
      const int n = n0 + 32 * c;
      if (r >= a.M || n >= a.N) continue;
      if (kOut != kOutF32Part) {
        const size_t off = (size_t)r * a.ldc + (size_t)z * a.c_nz + n;
        store_bf16_32(a.c16 + off, v, a.N - n);
        if (kOut == kOutBf16HiLo) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] -= __bfloat162float(__float2bfloat16_rn(v[i]));
          store_bf16_32(a.c16lo + off, v, a.N - n);
        }
      } else {
        float* dst = a.c32 + ((size_t)z * a.M + r) * a.ldc + n;
        if (n + 32 <= a.N) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (n + i < a.N) dst[i] = v[i];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kGN);
  }
}

// bf16 copy of an fp32 array, 8 numbers per thread step (n % 8 == 0)
__global__ void to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    reinterpret_cast<uint4*>(out)[i] =
        make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                   *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
  }
}

// fp32 -> bf16 rounded value and bf16 rounded remainder, 8 numbers per step
__global__ void to_bf16_hilo_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ hi,
                                    __nv_bfloat16* __restrict__ lo, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t wh[4], wl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      const __nv_bfloat162 l = __floats2bfloat162_rn(x[2 * e] - __low2float(h), x[2 * e + 1] - __high2float(h));
      wh[e] = *reinterpret_cast<const uint32_t*>(&h);
      wl[e] = *reinterpret_cast<const uint32_t*>(&l);
    }
    reinterpret_cast<uint4*>(hi)[i] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    reinterpret_cast<uint4*>(lo)[i] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
}

// W^UV [H * d_h, d_c] -> per head [d_c, d_h]: t[h][c][v] = w[h * d_h + v][c]
__global__ void transpose_heads_kernel(const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ t,
                                       int d_h, int d_c) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int h = blockIdx.z, v0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const __nv_bfloat16* src = w + (size_t)h * d_h * d_c;
  __nv_bfloat16* dst = t + (size_t)h * d_c * d_h;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int v = v0 + i, c = c0 + threadIdx.x;
    if (v < d_h && c < d_c) tile[i][threadIdx.x] = src[(size_t)v * d_c + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, v = v0 + threadIdx.x;
    if (v < d_h && c < d_c) dst[(size_t)c * d_h + v] = tile[threadIdx.x][i];
  }
}

// out = sum over the S partial sums, in split order (n4 float4 per partial)
__global__ void sum_splits_kernel(const float* __restrict__ part, int S, size_t n4, float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < S; ++s) {
      const float4 p = reinterpret_cast<const float4*>(part)[(size_t)s * n4 + i];
      acc.x += p.x;
      acc.y += p.y;
      acc.z += p.z;
      acc.w += p.w;
    }
    reinterpret_cast<float4*>(out)[i] = acc;
  }
}

// a row-major bf16 matrix [rows, cols] as a 2-D tensor map with box {64, box_rows}
cudaError_t bf16_map(TensorMapEncodeFn enc, CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                     uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kGK, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kBatched, bool kSplitA, int kOut>
cudaError_t launch_gemm(const GemmArgs& g, const CUtensorMap& ta, const CUtensorMap& talo, const CUtensorMap& tb,
                        dim3 grid, cudaStream_t s) {
  constexpr int smem = GemmShape<kSplitA>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(gemm_tn_kernel<kBatched, kSplitA, kOut>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  gemm_tn_kernel<kBatched, kSplitA, kOut><<<grid, kGT, smem, s>>>(g, ta, talo, tb);
  return cudaGetLastError();
}

unsigned grid_for(size_t n) { return (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096); }

}  // namespace

MergedSplit merged_output_split(int N, int H, int d_c, int d, int num_sms) {
  MergedSplit sp{};
  const long long K = (long long)H * d_c;
  const long long tiles = (long long)((d + kGN - 1) / kGN) * ((N + kGM - 1) / kGM);
  const long long kblocks = (K + kGK - 1) / kGK;
  long long S = tiles > 0 ? num_sms / tiles : 1;
  S = S < 1 ? 1 : (S > kblocks ? kblocks : S);
  const long long kb_per = (kblocks + S - 1) / S;
  sp.k_split = (int)(kb_per * kGK);
  sp.splits = (int)((K + sp.k_split - 1) / sp.k_split);
  const size_t a_bytes = ((size_t)N * K * 2 + 255) & ~(size_t)255;
  sp.a_offset = 0;
  sp.part_offset = a_bytes;
  sp.workspace_bytes = a_bytes + (size_t)sp.splits * N * d * 4;
  return sp;
}

cudaError_t launch_merge_output_weights(const MergeWArgs& a, cudaStream_t s) {
  TensorMapEncodeFn enc = nullptr;
  cudaError_t e = tensor_map_encoder(&enc);
  if (e != cudaSuccess) return e;
  // W^UV per head transposed, [H][d_c][d_h], in a scratch buffer
  __nv_bfloat16* t = nullptr;
  e = cudaMallocAsync(reinterpret_cast<void**>(&t), (size_t)a.H * a.d_c * a.d_h * 2, s);
  if (e != cudaSuccess) return e;
  transpose_heads_kernel<<<dim3((a.d_c + 31) / 32, (a.d_h + 31) / 32, a.H), dim3(32, 8), 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.w_uv), t, a.d_h, a.d_c);
  e = cudaGetLastError();
  CUtensorMap ta, tb;
  if (e == cudaSuccess) e = bf16_map(enc, &ta, a.w_o, (uint64_t)a.H * a.d_h, (uint64_t)a.d, kGM);
  if (e == cudaSuccess) e = bf16_map(enc, &tb, t, (uint64_t)a.d_h, (uint64_t)a.H * a.d_c, kGN);
  if (e == cudaSuccess) {
    GemmArgs g{};
    g.M = a.d;
    g.N = a.d_c;
    g.K = a.d_h;
    g.a_kz = a.d_h;
    g.b_nz = a.d_c;
    g.c16 = static_cast<__nv_bfloat16*>(a.w_merged);
    g.ldc = a.H * a.d_c;
    g.c_nz = a.d_c;
    g.err = a.err;
    e = launch_gemm<true, false, kOutBf16>(g, ta, ta, tb, dim3((a.d_c + kGN - 1) / kGN, (a.d + kGM - 1) / kGM, a.H), s);
  }
  const cudaError_t e2 = cudaFreeAsync(t, s);
  return e != cudaSuccess ? e : e2;
}

cudaError_t launch_absorb_output_merged(const MergedOArgs& a, cudaStream_t s) {
  TensorMapEncodeFn enc = nullptr;
  cudaError_t e = tensor_map_encoder(&enc);
  if (e != cudaSuccess) return e;
  const MergedSplit& sp = a.split;
  const size_t K = (size_t)a.H * a.d_c;
  auto* a16 = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(a.workspace) + sp.a_offset);
  auto* part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + sp.part_offset);
  const size_t n8 = (size_t)a.N * K / 8;
  to_bf16_kernel<<<grid_for(n8), 256, 0, s>>>(a.o_lat, a16, n8);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap ta, tb;
  e = bf16_map(enc, &ta, a16, K, (uint64_t)a.N, kGM);
  if (e == cudaSuccess) e = bf16_map(enc, &tb, a.w_merged, K, (uint64_t)a.d, kGN);
  if (e != cudaSuccess) return e;
  GemmArgs g{};
  g.M = a.N;
  g.N = a.d;
  g.K = (int)K;
  g.k_split = sp.k_split;
  g.c32 = part;
  g.ldc = a.d;
  g.err = a.err;
  e = launch_gemm<false, false, kOutF32Part>(g, ta, ta, tb, dim3((a.d + kGN - 1) / kGN, (a.N + kGM - 1) / kGM, sp.splits), s);
  if (e != cudaSuccess) return e;
  const size_t n4 = (size_t)a.N * a.d / 4;
  sum_splits_kernel<<<grid_for(n4), 256, 0, s>>>(part, sp.splits, n4, a.out);
  return cudaGetLastError();
}

bool absorb_output_tc_ok(const AbsorbOArgs& a) {
  const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return a.dtype == BF16 && a.d_c % 64 == 0 && a.d_h % 8 == 0 && a.d % 4 == 0 && a.N >= 1 &&
         (a.N + kGM - 1) / kGM <= 65535 && a.H <= 65535 && al16(a.o_lat) && al16(a.w_uv) && al16(a.w_o) &&
         al16(a.out) && (long long)a.H * a.d_c <= (1LL << 30);
}

cudaError_t launch_absorb_output_tc(const AbsorbOArgs& a, unsigned* err, int num_sms, cudaStream_t s) {
  TensorMapEncodeFn enc = nullptr;
  cudaError_t e = tensor_map_encoder(&enc);
  if (e != cudaSuccess) return e;
  const size_t KC = (size_t)a.H * a.d_c, KV = (size_t)a.H * a.d_h;
  // o = W^UV o_lat is the A of the second product: its K split like the merged output's
  const MergedSplit sp = merged_output_split(a.N, a.H, a.d_h, a.d, num_sms);
  const size_t b_lat = ((size_t)a.N * KC * 2 + 255) & ~(size_t)255;   // one bf16 copy of o_lat
  const size_t b_o = ((size_t)a.N * KV * 2 + 255) & ~(size_t)255;     // one bf16 copy of o
  const size_t b_part = (size_t)sp.splits * a.N * a.d * 4;
  uint8_t* ws = nullptr;
  e = cudaMallocAsync(reinterpret_cast<void**>(&ws), 2 * b_lat + 2 * b_o + b_part, s);
  if (e != cudaSuccess) return e;
  auto* lat_hi = reinterpret_cast<__nv_bfloat16*>(ws);
  auto* lat_lo = reinterpret_cast<__nv_bfloat16*>(ws + b_lat);
  auto* o_hi = reinterpret_cast<__nv_bfloat16*>(ws + 2 * b_lat);
  auto* o_lo = reinterpret_cast<__nv_bfloat16*>(ws + 2 * b_lat + b_o);
  auto* part = reinterpret_cast<float*>(ws + 2 * b_lat + 2 * b_o);
  const size_t n8 = (size_t)a.N * KC / 8;
  to_bf16_hilo_kernel<<<grid_for(n8), 256, 0, s>>>(a.o_lat, lat_hi, lat_lo, n8);
  e = cudaGetLastError();
  CUtensorMap t_hi, t_lo, t_w;
  // o[n, h*d_h + v] = sum_c W^UV[h*d_h + v, c] o_lat[n, h*d_c + c]: batched over heads
  if (e == cudaSuccess) e = bf16_map(enc, &t_hi, lat_hi, KC, (uint64_t)a.N, kGM);
  if (e == cudaSuccess) e = bf16_map(enc, &t_lo, lat_lo, KC, (uint64_t)a.N, kGM);
  if (e == cudaSuccess) e = bf16_map(enc, &t_w, a.w_uv, (uint64_t)a.d_c, KV, kGN);
  if (e == cudaSuccess) {
    GemmArgs g{};
    g.M = a.N;
    g.N = a.d_h;
    g.K = a.d_c;
    g.a_kz = a.d_c;
    g.b_nz = a.d_h;
    g.c16 = o_hi;
    g.c16lo = o_lo;
    g.ldc = (int)KV;
    g.c_nz = a.d_h;
    g.err = err;
    e = launch_gemm<true, true, kOutBf16HiLo>(g, t_hi, t_lo, t_w,
                                              dim3((a.d_h + kGN - 1) / kGN, (a.N + kGM - 1) / kGM, a.H), s);
  }
  // out[n, j] = sum_k W^O[j, k] o[n, k]: K split across the grid, partials summed in order
  if (e == cudaSuccess) e = bf16_map(enc, &t_hi, o_hi, KV, (uint64_t)a.N, kGM);
  if (e == cudaSuccess) e = bf16_map(enc, &t_lo, o_lo, KV, (uint64_t)a.N, kGM);
  if (e == cudaSuccess) e = bf16_map(enc, &t_w, a.w_o, KV, (uint64_t)a.d, kGN);
  if (e == cudaSuccess) {
    GemmArgs g{};
    g.M = a.N;
    g.N = a.d;
    g.K = (int)KV;
    g.k_split = sp.k_split;
    g.c32 = part;
    g.ldc = a.d;
    g.err = err;
    e = launch_gemm<false, true, kOutF32Part>(g, t_hi, t_lo, t_w,
                                              dim3((a.d + kGN - 1) / kGN, (a.N + kGM - 1) / kGM, sp.splits), s);
  }
  if (e == cudaSuccess) {
    const size_t n4 = (size_t)a.N * a.d / 4;
    sum_splits_kernel<<<grid_for(n4), 256, 0, s>>>(part, sp.splits, n4, a.out);
    e = cudaGetLastError();
  }
  const cudaError_t e2 = cudaFreeAsync(ws, s);
  return e != cudaSuccess ? e : e2;
}

}  // namespace mla
