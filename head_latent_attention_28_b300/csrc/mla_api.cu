// C ABI entry points: host-side argument checks, workspace carving, kernel
// selection, the per-device error word.  Declarations and the contract of
// each call are in include/mla.h.
#include <atomic>
#include <cmath>
#include <mutex>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "../../include/mla.h"

namespace {

__device__ unsigned int g_mla_error = 0;  // bits mla::kErr*

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

thread_local char g_last_cuda[256] = "";

// test hook of mla_test_set_wait_fault (zero: off)
std::atomic<int> g_test_skip_load{0};
// test knob of mla_test_force_splits (zero: off)
std::atomic<int> g_test_force_workers{0};
std::atomic<unsigned long long> g_test_wait_ns{0};

// Scratch of mla_decode_paged_noalloc: the split workspace (merge metadata,
// partial log-sum-exps and outputs) in a file-scope device array instead of
// caller memory.  64 MiB holds e.g. B = 32 sequences of 128 query rows with
// d_c = 512 at 74 split workers (49.6 MB: 27.9 MB of partials and 21.8 MB of
// the tensor-core kernel's message rings); larger shapes are rejected.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
__device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per
// device; the lookup may load the module, so make the first call before any
// stream capture).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

int note_cuda(cudaError_t e) {
  snprintf(g_last_cuda, sizeof(g_last_cuda), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

// Device address of the error word and SM count of the current device
// (looked up once per device; later calls read them without the lock).
std::atomic<bool> g_dev_ready[kMaxDevices];

cudaError_t device_info(unsigned** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_dev_ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_mla_error);
      if (e != cudaSuccess) return e;
      int n = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      g_num_sms[dev] = n;
      g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    g_dev_ready[dev].store(true, std::memory_order_release);
  }
  if (err) *err = g_err_ptr[dev];
  if (sms) *sms = g_num_sms[dev];
  return cudaSuccess;
}

bool dtype_ok(int d) { return d == MLA_F32 || d == MLA_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool decode_dims_ok(int B, int T_q, int H, int d_c, int d_r) {
  return B >= 1 && T_q >= 1 && H >= 1 && d_c >= 1 && d_c <= 512 && d_r >= 0 &&
         d_c + d_r <= 1024 && (long long)T_q * H <= (1 << 20);
}

int decode_workers(int dtype, int B, int T_q, int H, int d_c, int d_r, int sms) {
  (void)B;
  const int W = mla::tc_supported(dtype, H, T_q, d_c, d_r) ? mla::tc_workers(sms) : mla::generic_workers(sms);
  const int f = g_test_force_workers.load(std::memory_order_relaxed);
  return f > 0 && f < W ? f : W;
}

// the split partition's item cost for the kernel a shape selects (the
// CUDA-core kernel splits pages evenly)
int decode_item_cost(int dtype, int T_q, int H, int d_c, int d_r) {
  return mla::tc_supported(dtype, H, T_q, d_c, d_r) ? mla::tc_item_cost(T_q * H < 128 ? T_q * H : 128)
                                                     : 0;
}

// row groups of the kernel a shape selects: the tensor-core kernel takes at
// most 128 query rows per work item (G groups of SR rows), the CUDA-core
// kernel all rows of a sequence
void decode_row_groups(int dtype, int T_q, int H, int d_c, int d_r, int* G, int* SR) {
  const int rows = T_q * H;
  if (mla::tc_supported(dtype, H, T_q, d_c, d_r) && rows > 128) {
    *G = (rows + 127) / 128;
    *SR = 128;
  } else {
    *G = 1;
    *SR = rows;
  }
}

}  // namespace

extern "C" {

int mla_version(void) { return 100; }

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument (nothing launched)";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: unsupported shape or dtype";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call failed";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a device wait gave up";
    case MLA_ERR_BAD_INDEX: return "MLA_ERR_BAD_INDEX: block id or sequence length out of range";
    case MLA_ERR_BAD_RECORD: return "MLA_ERR_BAD_RECORD: the merge found no consistent split record";
    default: return "unknown mla status";
  }
}

const char* mla_last_cuda_error(void) { return g_last_cuda; }

int mla_check_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return note_cuda(e);
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_mla_error, sizeof(v));
  if (e != cudaSuccess) return note_cuda(e);
  if (v) {
    unsigned z = 0;
    e = cudaMemcpyToSymbol(g_mla_error, &z, sizeof(z));
    if (e != cudaSuccess) return note_cuda(e);
  }
  if (v & mla::kErrTimeout) return MLA_ERR_TIMEOUT;
  if (v & mla::kErrBadIndex) return MLA_ERR_BAD_INDEX;
  if (v & mla::kErrBadRecord) return MLA_ERR_BAD_RECORD;
  return MLA_OK;
}

int mla_test_force_splits(int num_workers) {
  if (num_workers < 0) return MLA_ERR_INVALID_ARG;
  g_test_force_workers.store(num_workers, std::memory_order_relaxed);
  return MLA_OK;
}

int mla_test_set_wait_fault(int skip_load, unsigned wait_us) {
  if (skip_load < 0) return MLA_ERR_INVALID_ARG;
  g_test_skip_load.store(skip_load, std::memory_order_relaxed);
  g_test_wait_ns.store(skip_load > 0 ? 1000ull * (wait_us ? wait_us : 1000u) : 0ull,
                       std::memory_order_relaxed);
  return MLA_OK;
}

int mla_cache_append(const void* c, const void* k_rope, int dtype_in,
                     const int32_t* seq_ids, const int32_t* positions, int n_new,
                     const int32_t* block_table, int B, int max_blocks_per_seq,
                     void* kv_cache, int cache_dtype, int num_blocks, int page_size,
                     int d_c, int d_r, float rope_base, void* stream) {
  if (n_new < 0 || B < 1 || d_c < 1 || d_r < 0 || (d_r & 1) || page_size != MLA_PAGE_SIZE ||
      max_blocks_per_seq < 1 || num_blocks < 1 || !dtype_ok(dtype_in) || !dtype_ok(cache_dtype) ||
      !(rope_base > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (n_new == 0) return MLA_OK;
  if (!c || (d_r > 0 && !k_rope) || !seq_ids || !positions || !block_table || !kv_cache)
    return MLA_ERR_INVALID_ARG;
  mla::AppendArgs a{c, k_rope, dtype_in, seq_ids, positions, n_new, block_table, B,
                    max_blocks_per_seq, kv_cache, cache_dtype, num_blocks, d_c, d_r,
                    rope_base, nullptr};
  cudaError_t e = device_info(&a.err, nullptr);
  if (e != cudaSuccess) return note_cuda(e);
  e = mla::launch_cache_append(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

int mla_absorb_query(const void* q_nope, const void* q_rope, const int32_t* positions,
                     const void* w_uk, int dtype, int N, int H, int d_h, int d_c,
                     int d_r, float rope_base, void* q_lat, int q_dtype, void* stream) {
  if (N < 0 || H < 1 || d_h < 1 || d_c < 1 || d_r < 0 || (d_r & 1) || !dtype_ok(dtype) ||
      !dtype_ok(q_dtype) || !(rope_base > 0.f) || d_h > 12288)
    return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!q_nope || (d_r > 0 && !q_rope) || !positions || !w_uk || !q_lat)
    return MLA_ERR_INVALID_ARG;
  mla::AbsorbQArgs a{q_nope, q_rope, positions, w_uk, dtype, N, H, d_h, d_c, d_r,
                     rope_base, q_lat, q_dtype, nullptr};
  if (H > 65535) return MLA_ERR_UNSUPPORTED;
  int sms = 0;
  cudaError_t ei = device_info(&a.err, &sms);
  if (ei != cudaSuccess) return note_cuda(ei);
  cudaError_t e = mla::launch_absorb_query(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

int mla_absorb_output(const float* o_lat, const void* w_uv, const void* w_o, int dtype,
                      int N, int H, int d_h, int d_c, int d, float* out, void* stream) {
  if (N < 0 || H < 1 || d_h < 1 || d_c < 1 || d < 1 || !dtype_ok(dtype) ||
      (long long)H * d_h > 32768)
    return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!o_lat || !w_uv || !w_o || !out) return MLA_ERR_INVALID_ARG;
  mla::AbsorbOArgs a{o_lat, w_uv, w_o, dtype, N, H, d_h, d_c, d, out};
  cudaError_t e;
  if (mla::absorb_output_tc_ok(a)) {
    unsigned* err = nullptr;
    int sms = 0;
    e = device_info(&err, &sms);
    if (e != cudaSuccess) return note_cuda(e);
    e = mla::launch_absorb_output_tc(a, err, sms, static_cast<cudaStream_t>(stream));
  } else {
    e = mla::launch_absorb_output(a, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

namespace {
bool merged_dims_ok(int H, int d_c, int d) {
  return H >= 1 && d_c >= 8 && d_c % 8 == 0 && d >= 4 && d % 4 == 0 && (long long)H * d_c <= (1LL << 30) &&
         d <= (1 << 24);
}
}  // namespace

int mla_merge_output_weights(const void* w_uv, const void* w_o, int dtype, int H, int d_h, int d_c, int d,
                             void* w_merged, void* stream) {
  if (!merged_dims_ok(H, d_c, d) || d_h < 1 || !dtype_ok(dtype) || (long long)H * d_h > (1LL << 30))
    return MLA_ERR_INVALID_ARG;
  if (!w_uv || !w_o || !w_merged || !aligned16(w_uv) || !aligned16(w_o) || !aligned16(w_merged)) return MLA_ERR_INVALID_ARG;
  if (dtype != MLA_BF16 || d_h % 64 != 0 || H > 65535) return MLA_ERR_UNSUPPORTED;
  mla::MergeWArgs a{w_uv, w_o, H, d_h, d_c, d, w_merged, nullptr};
  cudaError_t e = device_info(&a.err, nullptr);
  if (e != cudaSuccess) return note_cuda(e);
  e = mla::launch_merge_output_weights(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

size_t mla_absorb_output_merged_workspace_size(int N, int H, int d_c, int d) {
  if (N < 1 || !merged_dims_ok(H, d_c, d)) return 0;
  int sms = 0;
  if (device_info(nullptr, &sms) != cudaSuccess) return 0;
  return mla::merged_output_split(N, H, d_c, d, sms).workspace_bytes;
}

int mla_absorb_output_merged(const float* o_lat, const void* w_merged, int dtype, int N, int H, int d_c, int d,
                             void* workspace, size_t workspace_bytes, float* out, void* stream) {
  if (N < 0 || !merged_dims_ok(H, d_c, d) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!o_lat || !w_merged || !out || !aligned16(o_lat) || !aligned16(w_merged) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  if (dtype != MLA_BF16 || (long long)(N + 127) / 128 > 65535) return MLA_ERR_UNSUPPORTED;
  mla::MergedOArgs a{o_lat, w_merged, N, H, d_c, d, workspace, {}, out, nullptr};
  int sms = 0;
  cudaError_t e = device_info(&a.err, &sms);
  if (e != cudaSuccess) return note_cuda(e);
  a.split = mla::merged_output_split(N, H, d_c, d, sms);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < a.split.workspace_bytes)
    return MLA_ERR_WORKSPACE;
  e = mla::launch_absorb_output_merged(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

size_t mla_decode_workspace_size(int B, int T_q, int H, int d_c, int d_r, int dtype) {
  if (!decode_dims_ok(B, T_q, H, d_c, d_r) || !dtype_ok(dtype)) return 0;
  int sms = 0;
  if (device_info(nullptr, &sms) != cudaSuccess) return 0;
  const int W = decode_workers(dtype, B, T_q, H, d_c, d_r, sms);
  int G = 1, SR = 1;
  decode_row_groups(dtype, T_q, H, d_c, d_r, &G, &SR);
  if ((long long)B * G > (1 << 30)) return 0;
  const size_t msg = mla::tc_supported(dtype, H, T_q, d_c, d_r) ? mla::tc_msg_bytes_per_worker() : 0;
  return mla::ws_layout(B * G, SR, d_c, W, msg).total;
}

int mla_decode_split_plan(const int32_t* seqlens_host, int B, int T_q, int max_blocks_per_seq,
                          int num_workers, int item_cost, int32_t* first_worker,
                          int32_t* last_worker, int64_t* total_pages) {
  if (!seqlens_host || !first_worker || !last_worker || B < 1 || T_q < 1 ||
      max_blocks_per_seq < 1 || num_workers < 1 || item_cost < 0 || item_cost > 1024)
    return MLA_ERR_INVALID_ARG;
  const long long cap = (long long)max_blocks_per_seq * MLA_PAGE_SIZE;
  long long T = 0, U = 0;
  for (int b = 0; b < B; ++b) {
    const long long L = seqlens_host[b];
    if (L >= T_q && L <= cap) {
      const long long P = (L + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
      T += P;
      U += item_cost + P;
    }
  }
  long long A = 0;   // first unit of the next valid sequence
  const int Wa = mla::part_active(U, num_workers, item_cost);
  for (int b = 0; b < B; ++b) {
    const long long L = seqlens_host[b];
    if (L >= T_q && L <= cap) {
      const long long P = (L + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
      first_worker[b] = mla::part_worker_of(U, Wa, A + item_cost);
      last_worker[b] = mla::part_worker_of(U, Wa, A + item_cost + P - 1);
      A += item_cost + P;
    } else {
      first_worker[b] = last_worker[b] = -1;
    }
  }
  if (total_pages) *total_pages = T;
  return MLA_OK;
}

int mla_decode_item_cost(int T_q, int H, int d_c, int d_r, int dtype) {
  if (!decode_dims_ok(1, T_q, H, d_c, d_r) || !dtype_ok(dtype)) return -1;
  return decode_item_cost(dtype, T_q, H, d_c, d_r);
}

int mla_decode_row_groups(int T_q, int H, int d_c, int d_r, int dtype) {
  if (!decode_dims_ok(1, T_q, H, d_c, d_r) || !dtype_ok(dtype)) return -1;
  int G = 1, SR = 1;
  decode_row_groups(dtype, T_q, H, d_c, d_r, &G, &SR);
  return G;
}

int mla_decode_path(int T_q, int H, int d_c, int d_r, int dtype) {
  if (!decode_dims_ok(1, T_q, H, d_c, d_r) || !dtype_ok(dtype)) return -1;
  return mla::tc_supported(dtype, H, T_q, d_c, d_r) ? 1 : 0;
}

int mla_decode_num_workers(int B, int T_q, int H, int d_c, int d_r, int dtype) {
  if (!decode_dims_ok(B, T_q, H, d_c, d_r) || !dtype_ok(dtype)) return 0;
  int sms = 0;
  if (device_info(nullptr, &sms) != cudaSuccess) return 0;
  return decode_workers(dtype, B, T_q, H, d_c, d_r, sms);
}

}  // extern "C"

namespace {

enum DecodeStage { kStagePartial = 1, kStageCombine = 2, kStageBoth = 3 };

int decode_impl(int stage, const void* q_lat, const void* kv_cache, int dtype,
                const int32_t* block_table, const int32_t* seqlens,
                int B, int T_q, int H, int d_c, int d_r, int page_size,
                int max_blocks_per_seq, int num_blocks, float softmax_scale, int causal,
                void* workspace, size_t workspace_bytes, float* o_lat, float* lse,
                void* stream) {
  if (!q_lat || !kv_cache || !block_table || !seqlens || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!decode_dims_ok(B, T_q, H, d_c, d_r) || !dtype_ok(dtype) || page_size != MLA_PAGE_SIZE ||
      max_blocks_per_seq < 1 || num_blocks < 1 || !(softmax_scale > 0.f) ||
      (long long)max_blocks_per_seq * MLA_PAGE_SIZE > (1LL << 30))
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_lat) || !aligned16(kv_cache) || !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  mla::DecodeArgs a{};
  int sms = 0;
  cudaError_t e = device_info(&a.err, &sms);
  if (e != cudaSuccess) return note_cuda(e);
  const bool tc = mla::tc_supported(dtype, H, T_q, d_c, d_r);
  a.W = decode_workers(dtype, B, T_q, H, d_c, d_r, sms);
  a.item_cost = decode_item_cost(dtype, T_q, H, d_c, d_r);
  decode_row_groups(dtype, T_q, H, d_c, d_r, &a.G, &a.SR);
  if ((long long)B * a.G > (1 << 30)) return MLA_ERR_INVALID_ARG;
  const mla::WsLayout L = mla::ws_layout(B * a.G, a.SR, d_c, a.W, tc ? mla::tc_msg_bytes_per_worker() : 0);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  a.q = q_lat; a.cache = kv_cache; a.block_table = block_table; a.seqlens = seqlens;
  a.dtype = dtype; a.B = B; a.T_q = T_q; a.H = H; a.d_c = d_c; a.d_r = d_r; a.D = d_c + d_r;
  a.max_blocks = max_blocks_per_seq; a.num_blocks = num_blocks;
  a.scale = softmax_scale; a.causal = causal ? 1 : 0;
  a.o = o_lat; a.lse = lse;
  a.meta = reinterpret_cast<int2*>(ws + L.meta_off);
  a.ws_lse = reinterpret_cast<float*>(ws + L.lse_off);
  a.ws_o = reinterpret_cast<float*>(ws + L.o_off);
  a.msg = reinterpret_cast<unsigned char*>(ws + L.msg_off);
  a.skip_load = g_test_skip_load.load(std::memory_order_relaxed);
  a.wait_ns = g_test_wait_ns.load(std::memory_order_relaxed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (stage & kStagePartial) {
    e = tc ? mla::launch_decode_tc(a, s) : mla::launch_decode_generic(a, s);
    if (e != cudaSuccess) return note_cuda(e);
  }
  if (stage & kStageCombine) {
    e = mla::launch_combine(a, s);
    if (e != cudaSuccess) return note_cuda(e);
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_paged(const void* q_lat, const void* kv_cache, int dtype,
                     const int32_t* block_table, const int32_t* seqlens,
                     int B, int T_q, int H, int d_c, int d_r, int page_size,
                     int max_blocks_per_seq, int num_blocks,
                     float softmax_scale, int causal,
                     void* workspace, size_t workspace_bytes,
                     float* o_lat, float* lse, void* stream) {
  return decode_impl(kStageBoth, q_lat, kv_cache, dtype, block_table, seqlens, B, T_q, H, d_c,
                     d_r, page_size, max_blocks_per_seq, num_blocks, softmax_scale, causal,
                     workspace, workspace_bytes, o_lat, lse, stream);
}

int mla_decode_paged_noalloc(const void* q_lat, const void* kv_cache, int dtype,
                             const int32_t* block_table, const int32_t* seqlens,
                             int B, int T_q, int H, int d_c, int d_r, int page_size,
                             int max_blocks_per_seq, int num_blocks,
                             float softmax_scale, int causal,
                             float* o_lat, float* lse, void* stream) {
  if (!decode_dims_ok(B, T_q, H, d_c, d_r) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_size(B, T_q, H, d_c, d_r, dtype);
  if (need == 0) return MLA_ERR_CUDA;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) return note_cuda(e);
  // nothing in the workspace has to start at zero: the partial pass writes
  // every merge record and part that the combine reads in the same call
  return decode_impl(kStageBoth, q_lat, kv_cache, dtype, block_table, seqlens, B, T_q, H, d_c,
                     d_r, page_size, max_blocks_per_seq, num_blocks, softmax_scale, causal, ws,
                     kNoAllocScratchBytes, o_lat, lse, stream);
}

int mla_decode_paged_partial(const void* q_lat, const void* kv_cache, int dtype,
                             const int32_t* block_table, const int32_t* seqlens,
                             int B, int T_q, int H, int d_c, int d_r, int page_size,
                             int max_blocks_per_seq, int num_blocks,
                             float softmax_scale, int causal,
                             void* workspace, size_t workspace_bytes,
                             float* o_lat, float* lse, void* stream) {
  return decode_impl(kStagePartial, q_lat, kv_cache, dtype, block_table, seqlens, B, T_q, H,
                     d_c, d_r, page_size, max_blocks_per_seq, num_blocks, softmax_scale, causal,
                     workspace, workspace_bytes, o_lat, lse, stream);
}

int mla_decode_combine(const void* q_lat, const void* kv_cache, int dtype,
                       const int32_t* block_table, const int32_t* seqlens,
                       int B, int T_q, int H, int d_c, int d_r, int page_size,
                       int max_blocks_per_seq, int num_blocks,
                       float softmax_scale, int causal,
                       void* workspace, size_t workspace_bytes,
                       float* o_lat, float* lse, void* stream) {
  return decode_impl(kStageCombine, q_lat, kv_cache, dtype, block_table, seqlens, B, T_q, H,
                     d_c, d_r, page_size, max_blocks_per_seq, num_blocks, softmax_scale, causal,
                     workspace, workspace_bytes, o_lat, lse, stream);
}


// ---------------------------------------------------------------------------
// One decode step: absorb the new queries, append the new tokens' rows, attend.
// ---------------------------------------------------------------------------
static size_t step_q_bytes(int B, int T_q, int H, int d_c, int d_r, int dtype) {
  const size_t es = dtype == MLA_BF16 ? 2 : 4;
  return mla::align_up((size_t)B * (size_t)T_q * (size_t)H * (size_t)(d_c + d_r) * es, 256);
}

size_t mla_decode_step_workspace_size(int B, int T_q, int H, int d_c, int d_r, int dtype) {
  const size_t dec = mla_decode_workspace_size(B, T_q, H, d_c, d_r, dtype);
  if (dec == 0) return 0;
  return step_q_bytes(B, T_q, H, d_c, d_r, dtype) + dec;
}

int mla_decode_step(const void* q_nope, const void* q_rope, const void* w_uk, int d_h,
                    const void* c_new, const void* k_rope_new, void* kv_cache, int dtype,
                    const int32_t* block_table, const int32_t* seqlens,
                    int B, int T_q, int H, int d_c, int d_r, int page_size,
                    int max_blocks_per_seq, int num_blocks, float softmax_scale, int causal,
                    float rope_base, void* workspace, size_t workspace_bytes,
                    float* o_lat, float* lse, void* stream) {
  if (!q_nope || (d_r > 0 && (!q_rope || !k_rope_new)) || !w_uk || !c_new || !kv_cache ||
      !block_table || !seqlens || !o_lat)
    return MLA_ERR_INVALID_ARG;
  if (!decode_dims_ok(B, T_q, H, d_c, d_r) || !dtype_ok(dtype) || d_h < 1 || d_h > 12288 ||
      (d_r & 1) || !(rope_base > 0.f) || H > 65535 || (long long)B * T_q > (1LL << 30))
    return MLA_ERR_INVALID_ARG;
  const size_t qb = step_q_bytes(B, T_q, H, d_c, d_r, dtype);
  const size_t need = mla_decode_step_workspace_size(B, T_q, H, d_c, d_r, dtype);
  if (need == 0) return MLA_ERR_CUDA;
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MLA_ERR_WORKSPACE;
  unsigned* err = nullptr;
  cudaError_t e = device_info(&err, nullptr);
  if (e != cudaSuccess) return note_cuda(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* q_lat = workspace;                       // [B, T_q, H, d_c + d_r] in the cache dtype
  const int N = B * T_q;
  // 1. q_lat = [W^UK^T q_nope ; RoPE(q_rope)] at the new tokens' positions
  mla::AbsorbQArgs aq{q_nope, q_rope, nullptr, w_uk, dtype, N, H, d_h, d_c, d_r,
                      rope_base, q_lat, dtype, err};
  aq.seqlens = seqlens;
  aq.T_q = T_q;
  aq.step = true;
  // 2. the new tokens' rows [c ; RoPE(k_rope)] into the cache (in the same
  //    kernel as 1 when the absorption runs on the tensor cores)
  mla::AppendArgs ap{c_new, k_rope_new, dtype, nullptr, nullptr, N, block_table, B,
                     max_blocks_per_seq, kv_cache, dtype, num_blocks, d_c, d_r, rope_base, err};
  ap.seqlens = seqlens;
  ap.T_q = T_q;
  ap.step = true;
  e = mla::launch_absorb_and_append(aq, ap, s);
  if (e != cudaSuccess) return note_cuda(e);
  // 3. attention over the cache, split pass and merge
  return decode_impl(kStageBoth, q_lat, kv_cache, dtype, block_table, seqlens, B, T_q, H, d_c,
                     d_r, page_size, max_blocks_per_seq, num_blocks, softmax_scale, causal,
                     static_cast<char*>(workspace) + qb, workspace_bytes - qb, o_lat, lse, stream);
}

int mla_prefill_kv_rows(int max_blocks_per_seq) {
  if (max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 24)) return 0;
  return mla::prefill_kv_rows(max_blocks_per_seq);
}

int mla_prefill_use_rebuild(int T_q, int L, int H, int d_c, int d_r, int d_h, int dtype) {
  if (T_q < 1 || L < T_q || H < 1 || d_c < 1 || d_r < 0 || d_h < 1 || !dtype_ok(dtype)) return -1;
  if (!mla::prefill_supported(dtype, d_c, d_r, d_h) || !mla::tc_supported(dtype, H, T_q, d_c, d_r))
    return 0;
  // Whole-GPU costs measured on B300 (H = 128): the absorbed decode streams
  // every page once per group of 128 query rows, ~2.9 us per group and 4096
  // rows (32 x 4096 rows: 91.9 us per step); the rebuild takes ~168 us per
  // 4096 rows at 128 heads; the attention over rebuilt keys runs at ~980
  // TFLOP/s.
  const double rows = (double)H * T_q;
  const double groups = std::ceil(rows / 128.0);
  const double absorbed_us = groups * (double)L * (2.9 / 4096.0);
  const double visible = (double)T_q * (L - T_q) + 0.5 * (double)T_q * (T_q + 1);
  const double rebuild_us = (double)L * H * (168.0 / (4096.0 * 128.0)) +
                            (double)H * visible * 640.0 / 980.0e6;
  return rebuild_us < absorbed_us ? 1 : 0;
}

int mla_prefill_kv(const void* kv_cache, int dtype, const int32_t* block_table,
                   const int32_t* seqlens, int B, int d_c, int d_r, int page_size,
                   int max_blocks_per_seq, int num_blocks, const void* w_uk, const void* w_uv,
                   int H, int d_h, void* k_nope, void* v, void* k_rope, void* stream) {
  return mla_prefill_kv_chunk(kv_cache, dtype, block_table, seqlens, B, d_c, d_r, page_size, max_blocks_per_seq,
                              num_blocks, w_uk, w_uv, H, d_h, 0, k_nope, v, k_rope, stream);
}

int mla_prefill_kv_chunk(const void* kv_cache, int dtype, const int32_t* block_table,
                         const int32_t* seqlens, int B, int d_c, int d_r, int page_size,
                         int max_blocks_per_seq, int num_blocks, const void* w_uk, const void* w_uv,
                         int H, int d_h, int T_new, void* k_nope, void* v, void* k_rope, void* stream) {
  if (T_new < 0) return MLA_ERR_INVALID_ARG;
  if (B < 0 || H < 1 || d_h < 1 || d_c < 1 || d_r < 0 || !dtype_ok(dtype) ||
      page_size != MLA_PAGE_SIZE || max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 24) ||
      num_blocks < 1)
    return MLA_ERR_INVALID_ARG;
  if (!mla::prefill_supported(dtype, d_c, d_r, d_h)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  const auto al16 = [](const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(kv_cache) || !block_table || !seqlens || !al16(w_uk) || !al16(w_uv) ||
      !al16(k_nope) || !al16(v) || !al16(k_rope))
    return MLA_ERR_INVALID_ARG;
  const int R = mla::prefill_kv_rows(max_blocks_per_seq);
  if (B > 65535 || H > 65535 * 8 || (long long)B * R * H >= (1LL << 31) ||
      (long long)num_blocks * MLA_PAGE_SIZE >= (1LL << 31) || (long long)B * R >= (1LL << 31))
    return MLA_ERR_UNSUPPORTED;
  mla::PrefillKvArgs a{kv_cache, block_table, seqlens, B, max_blocks_per_seq, num_blocks, d_c, d_r,
                       w_uk, w_uv, H, d_h, R, k_nope, v, k_rope, nullptr, T_new};
  cudaError_t e = device_info(&a.err, nullptr);
  if (e != cudaSuccess) return note_cuda(e);
  e = mla::launch_prefill_kv(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

int mla_prefill_attention(const void* q_nope, const void* q_rope, int dtype, const void* k_nope,
                          const void* v, const void* k_rope, const int32_t* seqlens, int B,
                          int T_q, int H, int d_h, int d_r, int max_blocks_per_seq,
                          float rope_base, float softmax_scale, float* o, float* lse,
                          void* stream) {
  if (B < 0 || T_q < 1 || H < 1 || d_h < 1 || d_r < 0 || !dtype_ok(dtype) ||
      max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 24) || !(rope_base > 0.f) ||
      !(softmax_scale > 0.f) || !(softmax_scale < 3.0e38f))
    return MLA_ERR_INVALID_ARG;
  if (!mla::prefill_supported(dtype, 512, d_r, d_h)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  const auto al16 = [](const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(q_nope) || !q_rope || !al16(k_nope) || !al16(v) || !al16(k_rope) || !seqlens ||
      !al16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_INVALID_ARG;
  const int R = mla::prefill_kv_rows(max_blocks_per_seq);
  if (B > 65535 || H > 65535 || (long long)B * T_q >= (1LL << 31) ||
      (long long)B * H * R >= (1LL << 31) ||
      (long long)(T_q + 127) / 128 > 0x7fffffffLL)
    return MLA_ERR_UNSUPPORTED;
  mla::PrefillAttnArgs a{q_nope, q_rope, k_nope, v, k_rope, seqlens, B, T_q, H, d_h, d_r, R,
                         max_blocks_per_seq * MLA_PAGE_SIZE, softmax_scale, rope_base, o, lse, nullptr};
  cudaError_t e = device_info(&a.err, nullptr);
  if (e != cudaSuccess) return note_cuda(e);
  e = mla::launch_prefill_attn(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}
}  // extern "C"
