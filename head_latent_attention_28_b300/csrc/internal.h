// Launchers shared between the translation units of the library (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

// cuTensorMapEncodeTiled from the driver, looked up once (decode_tc.cu)
using TensorMapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                       const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                       const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                       CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
cudaError_t tensor_map_encoder(TensorMapEncodeFn* fn);

// decode_generic.cu
int generic_workers(int num_sms);
cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s);

// decode_tc.cu (tensor-core path: bf16, D = 576, d_c = 512, H*T_q in [64, 128])
bool tc_supported(int dtype, int H, int T_q, int d_c, int d_r);
int tc_workers(int num_sms);
int tc_item_cost(int rows);   // the split partition's item cost C for this kernel
size_t tc_msg_bytes_per_worker();   // message ring per split worker, in the workspace
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s);

// Rotary frequencies as turns per position, base^(-2j/d_r) / (2 pi), in
// 64-bit fixed point (computed on the host in double precision by
// rope_freqs, append_absorb.cu): the angle of position s is then s * turn[j]
// modulo one turn, exact in integer arithmetic up to the rounding of
// turn[j], with no large angle to reduce.
constexpr int kAbMaxPairs = 256;             // rotary pairs (d_r / 2) the table holds
struct RopeFreqs {
  uint64_t turn[kAbMaxPairs];
};
RopeFreqs rope_freqs(float base, int d_r);
#ifdef __CUDACC__
// the angle of pair j at position pos, in half turns (angle / pi) in [-1, 1):
// the 64-bit product pos * turn[j] wraps around whole turns
__device__ __forceinline__ double rope_half_turns(const RopeFreqs& fr, int pos, int j) {
  return (double)(int64_t)((uint64_t)(int64_t)pos * fr.turn[j]) * 0x1p-63;
}
#endif

// append_absorb.cu
struct AppendArgs {
  const void* c; const void* k_rope; int dtype_in;
  const int32_t* seq_ids; const int32_t* positions; int n_new;
  const int32_t* block_table; int B, max_blocks;
  void* cache; int cache_dtype; int num_blocks;
  int d_c, d_r; float rope_base;
  unsigned* err;
  // decode-step mode (seq_ids == positions == nullptr): token i is query
  // token t = i % T_q of sequence b = i / T_q, at position seqlens[b] - T_q + t
  const int32_t* seqlens = nullptr;
  int T_q = 1;
  bool step = false;   // launched as a programmatic dependent inside mla_decode_step
};
cudaError_t launch_cache_append(const AppendArgs& a, cudaStream_t s);

struct AbsorbQArgs {
  const void* q_nope; const void* q_rope; const int32_t* positions; const void* w_uk;
  int dtype; int N, H, d_h, d_c, d_r; float rope_base; void* q_lat; int q_dtype;
  unsigned* err;   // device error word (timeouts of the tensor-core kernel)
  // decode-step mode (positions == nullptr): token n is query token
  // t = n % T_q of sequence b = n / T_q, at position seqlens[b] - T_q + t
  const int32_t* seqlens = nullptr;
  int T_q = 1;
  bool step = false;   // first kernel of mla_decode_step: lets its dependents launch early
};
cudaError_t launch_absorb_query(const AbsorbQArgs& a, cudaStream_t s);
// the first two stages of mla_decode_step (query absorption, cache append)
cudaError_t launch_absorb_and_append(const AbsorbQArgs& a, const AppendArgs& ap, cudaStream_t s);

struct AbsorbOArgs {
  const float* o_lat; const void* w_uv; const void* w_o; int dtype;
  int N, H, d_h, d_c, d; float* out;
};
cudaError_t launch_absorb_output(const AbsorbOArgs& a, cudaStream_t s);

// out_proj_tc.cu (output projections on the tensor cores; bf16 weights)
struct MergeWArgs {
  const void* w_uv; const void* w_o;   // [H * d_h, d_c], [d, H * d_h]
  int H, d_h, d_c, d;
  void* w_merged;                      // [d, H * d_c] (output)
  unsigned* err;
};
cudaError_t launch_merge_output_weights(const MergeWArgs& a, cudaStream_t s);
// split of the merged output's K = H * d_c across the grid, and its workspace:
// the bf16 copy of o_lat at a_offset, fp32 partial sums [splits][N][d] at part_offset
struct MergedSplit {
  int splits, k_split;
  size_t a_offset, part_offset, workspace_bytes;
};
MergedSplit merged_output_split(int N, int H, int d_c, int d, int num_sms);
struct MergedOArgs {
  const float* o_lat; const void* w_merged;   // [N, H, d_c], [d, H * d_c]
  int N, H, d_c, d;
  void* workspace; MergedSplit split;
  float* out;                                 // [N, d]
  unsigned* err;
};
cudaError_t launch_absorb_output_merged(const MergedOArgs& a, cudaStream_t s);
// the unmerged pair of projections (mla_absorb_output) on the tensor cores:
// bf16 weights, d_c % 64 == 0, d_h % 8 == 0, d % 4 == 0, 16-byte aligned
bool absorb_output_tc_ok(const AbsorbOArgs& a);
cudaError_t launch_absorb_output_tc(const AbsorbOArgs& a, unsigned* err, int num_sms, cudaStream_t s);

// prefill_tc.cu (materialised per-head keys and values; bf16, d_c = 512,
// d_h = 128, d_r = 64)
bool prefill_supported(int dtype, int d_c, int d_r, int d_h);
int prefill_kv_rows(int max_blocks);   // rows per sequence of the rebuilt K/V buffers
struct PrefillKvArgs {
  const void* cache; const int32_t* block_table; const int32_t* seqlens;
  int B, max_blocks, num_blocks, d_c, d_r;
  const void* w_uk; const void* w_uv;   // [H * d_h, d_c]
  int H, d_h;
  int R;                                // rows per sequence of the outputs
  void* k_nope; void* v;                // [B, H, R, d_h] (head-major)
  void* k_rope;                         // [B, R, d_r]
  unsigned* err;
  int T_new = 0;                        // > 0: only rows [L - T_new, L) (and zeros past L) are written
};
cudaError_t launch_prefill_kv(const PrefillKvArgs& a, cudaStream_t s);
struct PrefillAttnArgs {
  const void* q_nope; const void* q_rope;   // [B, T_q, H, d_h], [B, T_q, H, d_r] (unrotated)
  const void* k_nope; const void* v; const void* k_rope;   // as PrefillKvArgs
  const int32_t* seqlens;
  int B, T_q, H, d_h, d_r;
  int R;                                    // rows per sequence of the K/V buffers
  int max_len;                              // longest valid sequence (max_blocks * 64)
  float scale, rope_base;
  float* o;                                 // [B, T_q, H, d_h]
  float* lse;                               // [B, T_q, H] or nullptr
  unsigned* err;
};
cudaError_t launch_prefill_attn(const PrefillAttnArgs& a, cudaStream_t s);

}  // namespace mla
