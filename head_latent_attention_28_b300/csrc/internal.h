// Launchers shared between the translation units of the library (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

// decode_generic.cu
int generic_workers(int num_sms);
cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s);

// decode_tc.cu (tensor-core path: bf16, D = 576, d_c = 512, H*T_q in [64, 128])
bool tc_supported(int dtype, int H, int T_q, int d_c, int d_r);
int tc_workers(int num_sms);
int tc_item_cost(int rows);   // the split partition's item cost C for this kernel
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s);

// append_absorb.cu
struct AppendArgs {
  const void* c; const void* k_rope; int dtype_in;
  const int32_t* seq_ids; const int32_t* positions; int n_new;
  const int32_t* block_table; int B, max_blocks;
  void* cache; int cache_dtype; int num_blocks;
  int d_c, d_r; float rope_base;
  unsigned* err;
};
cudaError_t launch_cache_append(const AppendArgs& a, cudaStream_t s);

struct AbsorbQArgs {
  const void* q_nope; const void* q_rope; const int32_t* positions; const void* w_uk;
  int dtype; int N, H, d_h, d_c, d_r; float rope_base; void* q_lat; int q_dtype;
};
cudaError_t launch_absorb_query(const AbsorbQArgs& a, cudaStream_t s);

struct AbsorbOArgs {
  const float* o_lat; const void* w_uv; const void* w_o; int dtype;
  int N, H, d_h, d_c, d; float* out;
};
cudaError_t launch_absorb_output(const AbsorbOArgs& a, cudaStream_t s);

}  // namespace mla
