// CUDA-core MLA decode: any d_c <= 512, any d_r, float or bfloat16 inputs.
//
// Serves the shapes the tensor-core kernel does not take (few heads, float
// caches, odd widths) and is the reference-precision path: every product and
// sum is in float (FFMA), exp2 in float, no reduced-precision operands.
//
// Math per (sequence b, query row r = t*H + h): online softmax over 32-token
// tiles of the visible cache rows,
//   m' = max(m, max_s z_s),  p_s = 2^(z_s - m'),  l' = l 2^(m - m') + sum p_s,
//   O' = O 2^(m - m') + sum_s p_s C_s[0:d_c]
// with z_s = log2(e) * scale * q . C_s, so that at the end o = O / l and
// lse = ln 2 * (m + log2 l).  ("Attention, Part 2", absorbed path: scores
// over the latent and the rotary key, causal mask, softmax, latent value sum.)
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr int GT = 256;   // threads per CTA
constexpr int GRT = 16;   // query rows per CTA
constexpr int GTK = 32;   // cache tokens per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ int pages_of(int L, int T_q, int cap) {
  return (L >= T_q && L <= cap) ? (L + kPage - 1) / kPage : 0;
}

// block-wide exclusive scan of one int per thread (GT threads); returns the
// exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* scratch /*[GT/32 + 1]*/, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < GT / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < GT / 32) scratch[lane] = w;  // inclusive warp totals
    if (lane == GT / 32 - 1) scratch[GT / 32] = w;
  }
  __syncthreads();
  int warp_base = warp ? scratch[warp - 1] : 0;
  *total = scratch[GT / 32];
  int r = warp_base + x - v;
  __syncthreads();
  return r;
}

template <typename T>
__global__ void __launch_bounds__(GT) decode_generic_kernel(DecodeArgs a) {
  extern __shared__ float smem[];
  const int D = a.D, Dp = D + 1;
  float* q_s = smem;                  // [GRT][D]
  float* k_s = q_s + GRT * D;         // [GTK][Dp]
  float* p_s = k_s + GTK * Dp;        // [GRT][GTK]  scores, then probabilities
  float* alpha_s = p_s + GRT * GTK;   // [GRT]
  float* m_s = alpha_s + GRT;         // [GRT]  running max (log2 units)
  float* l_s = m_s + GRT;             // [GRT]  running sum
  __shared__ long long tok_off[GTK];  // element offset of each tile row, -1 = absent
  __shared__ int scan_tmp[GT / 32 + 1];
  __shared__ long long red_tmp[GT / 32];
  __shared__ int seg_start[GT];       // exclusive page prefix within the chunk
  __shared__ int seg_first, seg_last;

  const T* __restrict__ q = static_cast<const T*>(a.q);
  const T* __restrict__ cache = static_cast<const T*>(a.cache);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int w = blockIdx.x;
  const int rows = a.T_q * a.H;
  const int r0 = blockIdx.y * GRT;
  const int cap = a.max_blocks * kPage;
  const float sl2 = a.scale * kLog2e;

  // ---- pass 1: total cost units (and the error flag for invalid lengths)
  const int C = a.item_cost;
  long long mine = 0;
  bool bad = false;
  for (int b = tid; b < a.B; b += GT) {
    int L = a.seqlens[b];
    int P = pages_of(L, a.T_q, cap);
    bad |= (P == 0);
    mine += P > 0 ? C + P : 0;
  }
  if (bad && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(a.err, kErrBadIndex);
#pragma unroll
  for (int o = 16; o; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) red_tmp[warp] = mine;
  __syncthreads();
  long long U = 0;
  for (int i = 0; i < GT / 32; ++i) U += red_tmp[i];
  if (U == 0) return;
  const int Wa = part_active(U, a.W, C);
  if (w >= Wa) return;
  const long long x0 = part_begin(U, Wa, w), x1 = part_begin(U, Wa, w + 1);

  // ---- pass 2: walk sequences in chunks, process the ones with pages in [x0, x1)
  long long base = 0;
  for (int c0 = 0; c0 < a.B && base < x1; c0 += GT) {
    const int bq = c0 + tid;
    const int P = bq < a.B ? pages_of(a.seqlens[bq], a.T_q, cap) : 0;
    int chunk_total;
    const int excl = block_exclusive_scan(P > 0 ? C + P : 0, scan_tmp, &chunk_total);
    seg_start[tid] = excl;
    if (tid == 0) { seg_first = GT; seg_last = -1; }
    __syncthreads();
    {
      int j0, j1;
      part_pages(x0, x1, base + excl + C, P, &j0, &j1);
      if (P > 0 && j1 > j0) { atomicMin(&seg_first, tid); atomicMax(&seg_last, tid); }
    }
    __syncthreads();
    const int f = seg_first, l = seg_last;
    for (int i = f; i <= l; ++i) {
      const int b = c0 + i;
      const int L = a.seqlens[b];
      const int Pb = pages_of(L, a.T_q, cap);
      if (Pb == 0) continue;
      const long long Ab = base + seg_start[i] + C;   // unit of the first page
      int j0, j1;
      part_pages(x0, x1, Ab, Pb, &j0, &j1);
      if (j1 <= j0) continue;
      const bool whole = (j0 == 0 && j1 == Pb);
      if (j0 == 0 && blockIdx.y == 0 && tid == 0)
        a.meta[b] = make_int2(part_worker_of(U, Wa, Ab), part_worker_of(U, Wa, Ab + Pb - 1));
      const int tok0 = j0 * kPage;
      const int tok1 = min(j1 * kPage, L);

      // load this CTA's query rows
      __syncthreads();
      for (int i2 = tid; i2 < GRT * D; i2 += GT) {
        int rr = i2 / D, k = i2 - rr * D;
        int r = r0 + rr;
        q_s[i2] = r < rows ? load_as_float(q, ((size_t)b * rows + r) * D + k) : 0.f;
      }
      if (tid < GRT) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }
      float acc[GRT][2];
#pragma unroll
      for (int rr = 0; rr < GRT; ++rr) acc[rr][0] = acc[rr][1] = 0.f;

      for (int s0 = tok0; s0 < tok1; s0 += GTK) {
        __syncthreads();
        if (tid < GTK) {
          int s = s0 + tid;
          long long off = -1;
          if (s < tok1) {
            int blk = a.block_table[(size_t)b * a.max_blocks + s / kPage];
            if (blk >= 0 && blk < a.num_blocks) off = ((long long)blk * kPage + (s % kPage)) * D;
            else atomicOr(a.err, kErrBadIndex);
          }
          tok_off[tid] = off;
        }
        __syncthreads();
        for (int i2 = tid; i2 < GTK * D; i2 += GT) {
          int j = i2 / D, k = i2 - j * D;
          long long off = tok_off[j];
          k_s[j * Dp + k] = off >= 0 ? load_as_float(cache, (size_t)off + k) : 0.f;
        }
        __syncthreads();
        // scores: lane = token, rows warp and warp + 8
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int rr = warp + 8 * half;
          const int r = r0 + rr;
          const float* qr = q_s + rr * D;
          const float* kr = k_s + lane * Dp;
          float dot = 0.f;
          for (int k = 0; k < D; ++k) dot = fmaf(qr[k], kr[k], dot);
          const int s = s0 + lane;
          const int t = r < rows ? r / a.H : 0;
          const int lim = a.causal ? (L - a.T_q + t) : (L - 1);
          const bool vis = r < rows && s < tok1 && tok_off[lane] >= 0 && s <= lim;
          p_s[rr * GTK + lane] = vis ? dot * sl2 : -INFINITY;
        }
        __syncthreads();
        // online softmax: warp handles rows 2*warp, 2*warp + 1
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int rr = 2 * warp + half;
          float v = p_s[rr * GTK + lane];
          float mx = v;
#pragma unroll
          for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const float m_old = m_s[rr];
          const float m_new = fmaxf(m_old, mx);
          float p, alpha;
          if (m_new == -INFINITY) { p = 0.f; alpha = 1.f; }
          else { p = exp2f(v - m_new); alpha = exp2f(m_old - m_new); }
          float sum = p;
#pragma unroll
          for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          p_s[rr * GTK + lane] = p;
          __syncwarp();
          if (lane == 0) { alpha_s[rr] = alpha; m_s[rr] = m_new; l_s[rr] = l_s[rr] * alpha + sum; }
        }
        __syncthreads();
        // value sum over the first d_c numbers of each row
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = tid + cc * GT;
          if (c < a.d_c) {
#pragma unroll
            for (int rr = 0; rr < GRT; ++rr) {
              float x = acc[rr][cc] * alpha_s[rr];
              const float* pr = p_s + rr * GTK;
#pragma unroll 8
              for (int j = 0; j < GTK; ++j) x = fmaf(pr[j], k_s[j * Dp + c], x);
              acc[rr][cc] = x;
            }
          }
        }
      }
      __syncthreads();
      // epilogue
      const int slot = b + w;
#pragma unroll
      for (int rr = 0; rr < GRT; ++rr) {
        const int r = r0 + rr;
        if (r >= rows) break;
        const float lsum = l_s[rr], m = m_s[rr];
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const float lse = lsum > 0.f ? (m + log2f(lsum)) * kLn2 : -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = tid + cc * GT;
          if (c < a.d_c) {
            if (whole) a.o[((size_t)b * rows + r) * a.d_c + c] = acc[rr][cc] * inv;
            else a.ws_o[((size_t)slot * rows + r) * a.d_c + c] = acc[rr][cc] * inv;
          }
        }
        if (tid == 0) {
          if (whole) { if (a.lse) a.lse[(size_t)b * rows + r] = lse; }
          else a.ws_lse[(size_t)slot * rows + r] = lse;
        }
      }
    }
    base += chunk_total;
    __syncthreads();
  }
}

constexpr int CT = 256;  // combine threads
constexpr int CR = 4;    // rows per combine CTA

// Merge the partial softmax results of sequences split across workers:
// lse* = max_i lse_i, w_i = exp(lse_i - lse*) (0 for an empty part),
// o = sum_i w_i o_i / sum_i w_i, lse = lse* + ln sum_i w_i.
// The normalised weights of the CTA's rows are computed once into shared
// memory; the output is then a weighted sum of VEC-wide column groups
// (float4 when d_c and the output allow it; coalesced either way).
// Sequences with an invalid length get zero outputs here.
template <int VEC>
struct VecT { using T = float; };
template <>
struct VecT<4> { using T = float4; };
__device__ __forceinline__ void fma_vec(float w, float v, float& acc) { acc = fmaf(w, v, acc); }
__device__ __forceinline__ void fma_vec(float w, const float4& v, float4& acc) {
  acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
}
__device__ __forceinline__ void zero_vec(float& v) { v = 0.f; }
__device__ __forceinline__ void zero_vec(float4& v) { v = make_float4(0.f, 0.f, 0.f, 0.f); }

template <int VEC>
__global__ void __launch_bounds__(CT) combine_kernel(DecodeArgs a) {
  using V = typename VecT<VEC>::T;
  // launched as a programmatic dependent of the partial pass: wait until that
  // grid has completed and its writes are visible (no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ float wts[];            // [CR][nw] normalised weights
  // one virtual sequence (sequence b, row group g) per blockIdx.x: its rows
  // [g * SR, g * SR + rows_g) of the sequence, slots vb + w of the workspace
  const int vb = blockIdx.x;
  const int b = vb / a.G, g = vb - b * a.G;
  const int rows = a.T_q * a.H;
  const int rows_g = min(a.SR, rows - g * a.SR);
  const int r0 = blockIdx.y * CR;
  const int nr = min(CR, rows_g - r0);
  if (nr <= 0) return;
  const size_t orow0 = (size_t)b * rows + (size_t)g * a.SR;   // first output row of the group
  const int L = a.seqlens[b];
  const bool valid = L >= a.T_q && L <= a.max_blocks * kPage;
  const int dc4 = a.d_c / VEC;
  if (!valid) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(a.err, kErrBadIndex);
    V z;
    zero_vec(z);
    for (int idx = threadIdx.x; idx < nr * dc4; idx += CT) {
      const int rr = idx / dc4, c4 = idx - rr * dc4;
      reinterpret_cast<V*>(a.o + (orow0 + r0 + rr) * a.d_c)[c4] = z;
    }
    if (threadIdx.x < nr && a.lse) a.lse[orow0 + r0 + threadIdx.x] = 0.f;
    return;
  }
  const int2 m = a.meta[vb];
  if (m.x == m.y) return;  // finished by its only worker
  if (m.x < 0 || m.y < m.x || m.y >= a.W) {
    // no consistent merge record (the partial pass gave up before writing
    // it, or no partial pass ran): report and write zeros rather than follow it
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(a.err, kErrBadRecord);
    V z;
    zero_vec(z);
    for (int idx = threadIdx.x; idx < nr * dc4; idx += CT) {
      const int rr = idx / dc4, c4 = idx - rr * dc4;
      reinterpret_cast<V*>(a.o + (orow0 + r0 + rr) * a.d_c)[c4] = z;
    }
    return;
  }
  const int nw = m.y - m.x + 1;
  // weights: one warp per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int rr = warp; rr < nr; rr += CT / 32) {
    const int r = r0 + rr;
    float lmax = -INFINITY;
    for (int k = lane; k < nw; k += 32) lmax = fmaxf(lmax, a.ws_lse[(size_t)(vb + m.x + k) * a.SR + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    float sumw = 0.f;
    for (int k = lane; k < nw; k += 32) {
      const float lw = a.ws_lse[(size_t)(vb + m.x + k) * a.SR + r];
      const float wt = (lw == -INFINITY) ? 0.f : expf(lw - lmax);
      wts[rr * nw + k] = wt;
      sumw += wt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sumw += __shfl_xor_sync(0xffffffffu, sumw, o);
    const float inv = sumw > 0.f ? 1.f / sumw : 0.f;
    __syncwarp();
    for (int k = lane; k < nw; k += 32) wts[rr * nw + k] *= inv;
    if (lane == 0 && a.lse) a.lse[orow0 + r] = sumw > 0.f ? lmax + logf(sumw) : -INFINITY;
  }
  __syncthreads();
  // each thread keeps kOut outputs in registers and issues the loads of up
  // to kParts parts for all of them together (the parts are L2-resident:
  // this kernel is latency-bound, so loads in flight decide its time)
  constexpr int kOut = 2, kParts = 4;
  const int total = nr * dc4;
  for (int base = threadIdx.x; base < total; base += CT * kOut) {
    V acc[kOut];
    int off[kOut], wrow[kOut];
#pragma unroll
    for (int t = 0; t < kOut; ++t) {
      zero_vec(acc[t]);
      const int idx = min(base + t * CT, total - 1);
      const int rr = idx / dc4, c4 = idx - rr * dc4;
      off[t] = (r0 + rr) * dc4 + c4;   // V index within a [rows, d_c] slab
      wrow[t] = rr * nw;
    }
    for (int k0 = 0; k0 < nw; k0 += kParts) {
      V v[kParts][kOut];
#pragma unroll
      for (int kk = 0; kk < kParts; ++kk) {
        const int k = min(k0 + kk, nw - 1);
        const V* part = reinterpret_cast<const V*>(a.ws_o + (size_t)(vb + m.x + k) * a.SR * a.d_c);
#pragma unroll
        for (int t = 0; t < kOut; ++t) v[kk][t] = part[off[t]];
      }
#pragma unroll
      for (int kk = 0; kk < kParts; ++kk)
        if (k0 + kk < nw) {
#pragma unroll
          for (int t = 0; t < kOut; ++t) fma_vec(wts[wrow[t] + k0 + kk], v[kk][t], acc[t]);
        }
    }
    V* out = reinterpret_cast<V*>(a.o + orow0 * a.d_c);
#pragma unroll
    for (int t = 0; t < kOut; ++t)
      if (base + t * CT < total) out[off[t]] = acc[t];
  }
}

size_t generic_smem_bytes(int D) {
  return sizeof(float) * ((size_t)GRT * D + (size_t)GTK * (D + 1) + GRT * GTK + 3 * GRT);
}

}  // namespace

int generic_workers(int num_sms) { return num_sms; }

cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = generic_smem_bytes(a.D);
  const int rows = a.T_q * a.H;
  dim3 grid(a.W, (rows + GRT - 1) / GRT);
  cudaError_t e;
  if (a.dtype == BF16) {
    e = cudaFuncSetAttribute(decode_generic_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    decode_generic_kernel<__nv_bfloat16><<<grid, GT, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(decode_generic_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    decode_generic_kernel<float><<<grid, GT, smem, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.B * a.G, (a.SR + CR - 1) / CR);
  // a sequence's parts come from at most W workers
  const size_t smem = sizeof(float) * (size_t)CR * (size_t)(a.W > 0 ? a.W : 1);
  const bool vec4 = a.d_c % 4 == 0 && (reinterpret_cast<uintptr_t>(a.o) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(a.ws_o) & 15u) == 0;
  auto kern = vec4 ? combine_kernel<4> : combine_kernel<1>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(CT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace mla
