// Cache append, query absorption and output absorption kernels.
//
// Each touches O(new tokens) data per step.  The append and the output
// absorption are written for exactness and simplicity (float accumulation,
// RoPE angles and rotations in double precision).  The query absorption,
// a per-head [tokens x d_h] . [d_h x 512] product that reads the whole W^UK
// once per step, has a tensor-core kernel for bf16 (below) and a plain one
// for everything else.
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace mla {

namespace {

template <typename T> __device__ __forceinline__ T cast_out(double x);
template <> __device__ __forceinline__ float cast_out<float>(double x) { return (float)x; }
template <> __device__ __forceinline__ __nv_bfloat16 cast_out<__nv_bfloat16>(double x) {
  return __float2bfloat16_rn((float)x);
}
template <typename T> __device__ __forceinline__ T cast_outf(float x);
template <> __device__ __forceinline__ float cast_outf<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 cast_outf<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// RoPE of one adjacent pair (x1, x2) at position pos, pair index j of d_r/2:
// rotate anticlockwise by pos * base^(-2j/d_r)  (RoFormer form).
__device__ __forceinline__ void rope_pair(double x1, double x2, int pos, int j, int d_r,
                                          double base, double* y1, double* y2) {
  const double theta = pow(base, -2.0 * (double)j / (double)d_r);
  double sn, cs;
  sincos((double)pos * theta, &sn, &cs);
  *y1 = x1 * cs - x2 * sn;
  *y2 = x1 * sn + x2 * cs;
}

// decode-step mode: token i is query token t = i % T_q of sequence b = i / T_q,
// at position seqlens[b] - T_q + t
__device__ __forceinline__ int step_position(const int32_t* seqlens, int T_q, int i, int* b) {
  *b = i / T_q;
  return seqlens[*b] - T_q + (i - *b * T_q);
}

// Row (seq, pos) of new token i <- [c ; RoPE_pos(k_rope)], written by nthr
// threads (index tid) together.  The angle is exact as a fraction of a turn;
// sine, cosine and the rotation run in float for a bf16 cache (whose rounding
// is far coarser) and in double for an fp32 one.
template <typename Tin, typename Tc>
__device__ __forceinline__ void write_cache_row(const AppendArgs& a, const RopeFreqs& fr, int i,
                                                int tid, int nthr) {
  int b, pos;
  if (a.seq_ids) {
    b = a.seq_ids[i];
    pos = a.positions[i];
  } else {
    pos = step_position(a.seqlens, a.T_q, i, &b);
  }
  const int D = a.d_c + a.d_r;
  if (b < 0 || b >= a.B || pos < 0 || pos >= a.max_blocks * kPage) {
    if (tid == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const int blk = a.block_table[(size_t)b * a.max_blocks + pos / kPage];
  if (blk < 0 || blk >= a.num_blocks) {
    if (tid == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const Tin* c = static_cast<const Tin*>(a.c) + (size_t)i * a.d_c;
  const Tin* kr = static_cast<const Tin*>(a.k_rope) + (size_t)i * a.d_r;
  Tc* row = static_cast<Tc*>(a.cache) + ((size_t)blk * kPage + pos % kPage) * D;
  if (nthr == 1 && sizeof(Tin) == 2 && sizeof(Tc) == 2 && a.d_c % 8 == 0 &&
      ((reinterpret_cast<uintptr_t>(c) | reinterpret_cast<uintptr_t>(row)) & 15u) == 0) {
    // one thread per row: the bf16 latent moves unchanged, 16 bytes at a time
    for (int k = 0; k < a.d_c / 8; ++k)
      reinterpret_cast<uint4*>(row)[k] = reinterpret_cast<const uint4*>(c)[k];
  } else {
    for (int k = tid; k < a.d_c; k += nthr) row[k] = cast_outf<Tc>(load_as_float(c, k));
  }
  for (int j = tid; j < a.d_r / 2; j += nthr) {
    const float x1 = load_as_float(kr, 2 * j), x2 = load_as_float(kr, 2 * j + 1);
    if (a.d_r / 2 > kAbMaxPairs) {
      double y1, y2;
      rope_pair(x1, x2, pos, j, a.d_r, (double)a.rope_base, &y1, &y2);
      row[a.d_c + 2 * j] = cast_out<Tc>(y1);
      row[a.d_c + 2 * j + 1] = cast_out<Tc>(y2);
    } else if (sizeof(Tc) == 2) {
      float sn, cs;
      sincospif((float)rope_half_turns(fr, pos, j), &sn, &cs);
      row[a.d_c + 2 * j] = cast_outf<Tc>(x1 * cs - x2 * sn);
      row[a.d_c + 2 * j + 1] = cast_outf<Tc>(x1 * sn + x2 * cs);
    } else {
      double sn, cs;
      sincospi(rope_half_turns(fr, pos, j), &sn, &cs);
      row[a.d_c + 2 * j] = cast_out<Tc>((double)x1 * cs - (double)x2 * sn);
      row[a.d_c + 2 * j + 1] = cast_out<Tc>((double)x1 * sn + (double)x2 * cs);
    }
  }
}

// One CTA per new token.
template <typename Tin, typename Tc>
__global__ void __launch_bounds__(128) cache_append_kernel(AppendArgs a, const __grid_constant__ RopeFreqs fr) {
  // inside mla_decode_step: the query absorption before this kernel must be
  // complete before this one is (the decode waits for this kernel only)
  if (a.step) asm volatile("griddepcontrol.wait;" ::: "memory");
  write_cache_row<Tin, Tc>(a, fr, blockIdx.x, threadIdx.x, blockDim.x);
}

// One CTA per (token n, head h):
//   q_lat[n,h,0:d_c] = W^UK_h^T q_nope[n,h,:],  q_lat[n,h,d_c:] = RoPE(q_rope[n,h,:]).
template <typename Tin, typename Tq>
__global__ void __launch_bounds__(128) absorb_query_kernel(AbsorbQArgs a) {
  extern __shared__ float qn[];  // [d_h]
  const int n = blockIdx.x, h = blockIdx.y;
  const int D = a.d_c + a.d_r;
  const Tin* q_nope = static_cast<const Tin*>(a.q_nope) + ((size_t)n * a.H + h) * a.d_h;
  const Tin* q_rope = static_cast<const Tin*>(a.q_rope) + ((size_t)n * a.H + h) * a.d_r;
  const Tin* w = static_cast<const Tin*>(a.w_uk) + (size_t)h * a.d_h * a.d_c;
  Tq* out = static_cast<Tq*>(a.q_lat) + ((size_t)n * a.H + h) * D;
  for (int d = threadIdx.x; d < a.d_h; d += blockDim.x) qn[d] = load_as_float(q_nope, d);
  __syncthreads();
  for (int c = threadIdx.x; c < a.d_c; c += blockDim.x) {
    float acc = 0.f;
    for (int d = 0; d < a.d_h; ++d) acc = fmaf(qn[d], load_as_float(w, (size_t)d * a.d_c + c), acc);
    out[c] = cast_outf<Tq>(acc);
  }
  int bq;
  const int pos = a.positions ? a.positions[n] : step_position(a.seqlens, a.T_q, n, &bq);
  for (int j = threadIdx.x; j < a.d_r / 2; j += blockDim.x) {
    double y1, y2;
    rope_pair(load_as_float(q_rope, 2 * j), load_as_float(q_rope, 2 * j + 1), pos, j, a.d_r,
              (double)a.rope_base, &y1, &y2);
    out[a.d_c + 2 * j] = cast_out<Tq>(y1);
    out[a.d_c + 2 * j + 1] = cast_out<Tq>(y2);
  }
}

// Tensor-core query absorption (bf16, d_c = 512, d_h = 64 or 128): one CTA
// per (head h, tile of 128 tokens).  TMA brings W^UK_h (d_h x 512, kept
// MN-major: eight 64-column chunks of d_h rows, SW128) and the tile's q_nope
// rows (K-major SW128, one 64-dim box per 64 of d_h) into shared memory; one
// thread issues tcgen05.mma with M = 128 tokens, N = 256, K = 16 into TMEM
// (all 512 fp32 columns); the four warps read their 32 tokens back (token r
// in TMEM lane r) and write q_lat with 16-byte stores, then rotate the rotary
// query.  Tokens past N are zero rows (TMA fill) and are not written.  Waits
// are bounded (2 s); on expiry the kernel sets MLA_ERR_TIMEOUT and writes
// nothing.
constexpr int kAbT = 128;                    // threads = tokens per CTA
constexpr int kAbSmem = 2 * 16384 + 8 * 128 * 128 + 1024;
constexpr uint64_t kAbWaitNs = 2000000000ull;

__device__ __forceinline__ void store32(float* dst, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}
__device__ __forceinline__ void store32(__nv_bfloat16* dst, const float (&v)[32]) {
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
}

template <typename Tq>
__global__ void __launch_bounds__(kAbT, 1)
absorb_query_tc_kernel(const AbsorbQArgs a, const __grid_constant__ CUtensorMap tm_qn,
                       const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ RopeFreqs fr,
                       const AppendArgs ap) {
  using namespace sm100;
  extern __shared__ uint8_t ab_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ab_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ uint64_t full, done;
  __shared__ uint32_t tbase;
  __shared__ int failed, never;
  // inside mla_decode_step the next kernel (the cache append) may launch now
  if (a.step) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.x, n0 = blockIdx.y * kAbT;
  const int kb = a.d_h / 64;                        // 64-dim boxes of q_nope along K
  const uint32_t wchunk = (uint32_t)a.d_h * 128;    // bytes of one 64-column chunk of W^UK_h
  uint8_t* sa = smem;                               // q_nope tile
  uint8_t* sw = smem + 2 * 16384;                   // W^UK_h
  if (threadIdx.x == 0) {
    failed = 0;
    never = 0;
    mbar_init(&full, 1);
    mbar_init(&done, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 0) tmem_alloc(&tbase, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(&full, (uint32_t)kb * 16384 + 8 * wchunk);
    for (int k = 0; k < kb; ++k) tma_load_3d(sa + k * 16384, &tm_qn, &full, 64 * k, h, n0, pol);
    for (int j = 0; j < 8; ++j) tma_load_2d(sw + j * wchunk, &tm_w, &full, 64 * j, h * a.d_h, pol);
    if (mbar_wait(&full, 0, &never, kAbWaitNs)) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_f32(128, 256, 0, 1);   // A K-major, B MN-major
      for (int nh = 0; nh < 2; ++nh)
        for (int kk = 0; kk < a.d_h / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(smem_u32(sa + (kk >> 2) * 16384 + (kk & 3) * 32), 16, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(sw + nh * 4 * wchunk + kk * 2048), wchunk, 1024);
          mma_ss(tmem + nh * 256, ad, bd, id, kk > 0 ? 1 : 0);
        }
      mma_commit(&done);
    } else {
      failed = 1;
      atomicOr(a.err, kErrTimeout);
      mbar_wait(&full, 0, &never, kAbWaitNs);   // the copies in flight land before the CTA exits
    }
  }
  __syncwarp();
  // inside mla_decode_step these CTAs also append the new tokens' cache rows
  // while the tensor core works: token n0 + t goes to the CTA of head
  // t mod H, whose threads write its row together (the same arithmetic as
  // the append kernel)
  if (ap.n_new > 0)
    for (int t = h; t < kAbT && n0 + t < ap.n_new; t += a.H)
      write_cache_row<__nv_bfloat16, __nv_bfloat16>(ap, fr, n0 + t, threadIdx.x, kAbT);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&done, 0, &failed, kAbWaitNs));
  tc_fence_after();
  const int n = n0 + threadIdx.x;                   // the token of this TMEM lane
  const int D = a.d_c + a.d_r;
  Tq* out = static_cast<Tq*>(a.q_lat) + ((size_t)(n < a.N ? n : 0) * a.H + h) * D;
  if (ok) {
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
#pragma unroll 1
    for (int c = 0; c < 16; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_off + 32 * c, v);
      tmem_ld_wait();
      if (n < a.N) store32(out + 32 * c, v);
    }
    // rotary dims: the angle as a fraction of a turn in [-1/2, 1/2), from the
    // 64-bit product position * turn[j] (its wrap-around drops the whole
    // turns); sine, cosine and the rotation in float
    if (n < a.N) {
      const __nv_bfloat16* q_rope =
          static_cast<const __nv_bfloat16*>(a.q_rope) + ((size_t)n * a.H + h) * a.d_r;
      int bq;
      const int p = a.positions ? a.positions[n] : step_position(a.seqlens, a.T_q, n, &bq);
      const uint64_t pos = (uint64_t)(int64_t)p;   // two's complement: modular product
      for (int j = 0; j < a.d_r / 2; ++j) {
        const float half_turns = (float)(int64_t)(pos * fr.turn[j]) * 0x1p-63f;   // angle / pi
        float sn, cs;
        sincospif(half_turns, &sn, &cs);
        const float x1 = load_as_float(q_rope, 2 * j), x2 = load_as_float(q_rope, 2 * j + 1);
        out[a.d_c + 2 * j] = cast_outf<Tq>(x1 * cs - x2 * sn);
        out[a.d_c + 2 * j + 1] = cast_outf<Tq>(x1 * sn + x2 * cs);
      }
    }
  } else if (threadIdx.x == 0) {
    atomicOr(a.err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

bool absorb_tc_ok(const AbsorbQArgs& a) {
  const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return a.dtype == BF16 && a.d_c == 512 && (a.d_h == 64 || a.d_h == 128) && a.N >= 1 &&
         a.d_r / 2 <= kAbMaxPairs && a.err != nullptr && al16(a.q_nope) && al16(a.w_uk) &&
         al16(a.q_lat) && (long long)a.H * a.d_h < (1LL << 31) && (long long)a.N <= 65535LL * kAbT;
}

cudaError_t launch_absorb_query_tc(const AbsorbQArgs& a, const AppendArgs& ap, cudaStream_t s) {
  TensorMapEncodeFn enc = nullptr;
  cudaError_t e = tensor_map_encoder(&enc);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_qn, tm_w;
  {
    // q_nope [N, H, d_h] as a 3-D tensor: box of 64 dims x 1 head x 128 tokens
    cuuint64_t dims[3] = {(cuuint64_t)a.d_h, (cuuint64_t)a.H, (cuuint64_t)a.N};
    cuuint64_t strides[2] = {(cuuint64_t)a.d_h * 2, (cuuint64_t)a.H * a.d_h * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kAbT};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_qn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q_nope), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // w_uk [H * d_h, 512]: box of 64 columns x d_h rows (one head)
    cuuint64_t dims[2] = {(cuuint64_t)a.d_c, (cuuint64_t)a.H * a.d_h};
    cuuint64_t strides[1] = {(cuuint64_t)a.d_c * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)a.d_h};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.w_uk), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const RopeFreqs fr = rope_freqs(a.rope_base, a.d_r);
  dim3 grid(a.H, (a.N + kAbT - 1) / kAbT), block(kAbT);
  if (a.q_dtype == F32) {
    e = cudaFuncSetAttribute(absorb_query_tc_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAbSmem);
    if (e != cudaSuccess) return e;
    absorb_query_tc_kernel<float><<<grid, block, kAbSmem, s>>>(a, tm_qn, tm_w, fr, ap);
  } else {
    e = cudaFuncSetAttribute(absorb_query_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAbSmem);
    if (e != cudaSuccess) return e;
    absorb_query_tc_kernel<__nv_bfloat16><<<grid, block, kAbSmem, s>>>(a, tm_qn, tm_w, fr, ap);
  }
  return cudaGetLastError();
}

constexpr int AO_T = 256;    // threads
constexpr int AO_J = 256;    // output columns per CTA

// CTA (n, column chunk): o[n] = per-head W^UV_h o_lat[n,h] into shared memory,
// then out[n, j] = W^O[j, :] . o[n] for the chunk's columns.
template <typename Tw>
__global__ void __launch_bounds__(AO_T) absorb_output_kernel(AbsorbOArgs a) {
  extern __shared__ float o_s[];  // [H * d_h]
  const int n = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int HD = a.H * a.d_h;
  const Tw* w_uv = static_cast<const Tw*>(a.w_uv);
  const Tw* w_o = static_cast<const Tw*>(a.w_o);
  for (int k = warp; k < HD; k += AO_T / 32) {
    const int h = k / a.d_h;
    const float* ol = a.o_lat + ((size_t)n * a.H + h) * a.d_c;
    const Tw* wr = w_uv + (size_t)k * a.d_c;
    float acc = 0.f;
    for (int c = lane; c < a.d_c; c += 32) acc = fmaf(load_as_float(wr, c), ol[c], acc);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) o_s[k] = acc;
  }
  __syncthreads();
  const int j_end = min(a.d, (int)(blockIdx.y + 1) * AO_J);
  for (int j = blockIdx.y * AO_J + warp; j < j_end; j += AO_T / 32) {
    const Tw* wr = w_o + (size_t)j * HD;
    float acc = 0.f;
    for (int k = lane; k < HD; k += 32) acc = fmaf(load_as_float(wr, k), o_s[k], acc);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.out[(size_t)n * a.d + j] = acc;
  }
}

}  // namespace

RopeFreqs rope_freqs(float base, int d_r) {
  RopeFreqs fr{};
  for (int j = 0; j < d_r / 2 && j < kAbMaxPairs; ++j) {
    const double turns = std::pow((double)base, -2.0 * (double)j / (double)d_r) /
                         6.283185307179586476925286766559;   // < 1
    fr.turn[j] = (uint64_t)std::ldexp(turns, 64);
  }
  return fr;
}

cudaError_t launch_cache_append(const AppendArgs& a, cudaStream_t s) {
  if (a.n_new == 0) return cudaSuccess;
  const RopeFreqs fr = rope_freqs(a.rope_base, a.d_r);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_new);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = a.step ? 1 : 0;
  if (a.dtype_in == F32 && a.cache_dtype == F32)
    return cudaLaunchKernelEx(&cfg, cache_append_kernel<float, float>, a, fr);
  if (a.dtype_in == F32) return cudaLaunchKernelEx(&cfg, cache_append_kernel<float, __nv_bfloat16>, a, fr);
  if (a.cache_dtype == F32) return cudaLaunchKernelEx(&cfg, cache_append_kernel<__nv_bfloat16, float>, a, fr);
  return cudaLaunchKernelEx(&cfg, cache_append_kernel<__nv_bfloat16, __nv_bfloat16>, a, fr);
}

cudaError_t launch_absorb_query(const AbsorbQArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (absorb_tc_ok(a)) {
    AppendArgs none{};
    none.n_new = 0;
    return launch_absorb_query_tc(a, none, s);
  }
  dim3 grid(a.N, a.H), block(128);
  size_t smem = sizeof(float) * a.d_h;
  if (a.dtype == F32 && a.q_dtype == F32) absorb_query_kernel<float, float><<<grid, block, smem, s>>>(a);
  else if (a.dtype == F32) absorb_query_kernel<float, __nv_bfloat16><<<grid, block, smem, s>>>(a);
  else if (a.q_dtype == F32) absorb_query_kernel<__nv_bfloat16, float><<<grid, block, smem, s>>>(a);
  else absorb_query_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_absorb_and_append(const AbsorbQArgs& a, const AppendArgs& ap, cudaStream_t s) {
  // one kernel when the absorption runs on the tensor cores and the cache is
  // bf16 like the query; otherwise the two kernels, the append as a
  // programmatic dependent of the absorption
  if (absorb_tc_ok(a) && a.q_dtype == BF16 && ap.dtype_in == BF16 && ap.cache_dtype == BF16 &&
      ap.n_new == a.N && ap.d_c == a.d_c && ap.d_r == a.d_r && ap.rope_base == a.rope_base)
    return launch_absorb_query_tc(a, ap, s);
  cudaError_t e = launch_absorb_query(a, s);
  if (e != cudaSuccess) return e;
  return launch_cache_append(ap, s);
}

cudaError_t launch_absorb_output(const AbsorbOArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  dim3 grid(a.N, (a.d + AO_J - 1) / AO_J), block(AO_T);
  size_t smem = sizeof(float) * (size_t)a.H * a.d_h;
  cudaError_t e;
  if (a.dtype == F32) {
    e = cudaFuncSetAttribute(absorb_output_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    absorb_output_kernel<float><<<grid, block, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(absorb_output_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    absorb_output_kernel<__nv_bfloat16><<<grid, block, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mla
