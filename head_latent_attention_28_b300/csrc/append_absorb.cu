// Cache append, query absorption and output absorption kernels.
//
// None of these is on the per-step hot loop (each touches O(new tokens)
// data), so they are written for exactness and simplicity: float
// accumulation, RoPE angles and rotations in double precision.
#include "common.cuh"
#include "internal.h"

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

// One CTA per new token: row (seq, pos) <- [c ; RoPE_pos(k_rope)].
template <typename Tin, typename Tc>
__global__ void __launch_bounds__(128) cache_append_kernel(AppendArgs a) {
  const int i = blockIdx.x;
  const int b = a.seq_ids[i], pos = a.positions[i];
  const int D = a.d_c + a.d_r;
  if (b < 0 || b >= a.B || pos < 0 || pos >= a.max_blocks * kPage) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const int blk = a.block_table[(size_t)b * a.max_blocks + pos / kPage];
  if (blk < 0 || blk >= a.num_blocks) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const Tin* c = static_cast<const Tin*>(a.c) + (size_t)i * a.d_c;
  const Tin* kr = static_cast<const Tin*>(a.k_rope) + (size_t)i * a.d_r;
  Tc* row = static_cast<Tc*>(a.cache) + ((size_t)blk * kPage + pos % kPage) * D;
  for (int k = threadIdx.x; k < a.d_c; k += blockDim.x)
    row[k] = cast_outf<Tc>(load_as_float(c, k));
  for (int j = threadIdx.x; j < a.d_r / 2; j += blockDim.x) {
    double y1, y2;
    rope_pair(load_as_float(kr, 2 * j), load_as_float(kr, 2 * j + 1), pos, j, a.d_r,
              (double)a.rope_base, &y1, &y2);
    row[a.d_c + 2 * j] = cast_out<Tc>(y1);
    row[a.d_c + 2 * j + 1] = cast_out<Tc>(y2);
  }
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
  const int pos = a.positions[n];
  for (int j = threadIdx.x; j < a.d_r / 2; j += blockDim.x) {
    double y1, y2;
    rope_pair(load_as_float(q_rope, 2 * j), load_as_float(q_rope, 2 * j + 1), pos, j, a.d_r,
              (double)a.rope_base, &y1, &y2);
    out[a.d_c + 2 * j] = cast_out<Tq>(y1);
    out[a.d_c + 2 * j + 1] = cast_out<Tq>(y2);
  }
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

cudaError_t launch_cache_append(const AppendArgs& a, cudaStream_t s) {
  if (a.n_new == 0) return cudaSuccess;
  dim3 grid(a.n_new), block(128);
  if (a.dtype_in == F32 && a.cache_dtype == F32) cache_append_kernel<float, float><<<grid, block, 0, s>>>(a);
  else if (a.dtype_in == F32) cache_append_kernel<float, __nv_bfloat16><<<grid, block, 0, s>>>(a);
  else if (a.cache_dtype == F32) cache_append_kernel<__nv_bfloat16, float><<<grid, block, 0, s>>>(a);
  else cache_append_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_absorb_query(const AbsorbQArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  dim3 grid(a.N, a.H), block(128);
  size_t smem = sizeof(float) * a.d_h;
  if (a.dtype == F32 && a.q_dtype == F32) absorb_query_kernel<float, float><<<grid, block, smem, s>>>(a);
  else if (a.dtype == F32) absorb_query_kernel<float, __nv_bfloat16><<<grid, block, smem, s>>>(a);
  else if (a.q_dtype == F32) absorb_query_kernel<__nv_bfloat16, float><<<grid, block, smem, s>>>(a);
  else absorb_query_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, smem, s>>>(a);
  return cudaGetLastError();
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
