// Internal declarations shared by the host and CUDA translation units of libtq.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda_runtime_api.h>

#include "tq.h"

namespace tq {

// Records a formatted error message for tq_last_error() and returns `st`.
tq_status fail(tq_status st, const char* fmt, ...);
void clear_error();

// Adds one to the count tq_launch_count() reports; called after each kernel launch.
void count_launch();

// Host-side validation of a descriptor.  Returns TQ_OK or an error (message set).
// need_data = false skips the device-pointer checks (sizes only).
tq_status check_desc(const tq_cache_desc* desc, bool need_data = true);

// Bytes of a K (which = 0) or V (which = 1) page of a valid descriptor.
size_t page_bytes_of(const tq_cache_desc& d, int which);

// Splits chosen when the caller passes 0: one chunk per decode warp of the GPU
// (warps = warps per decode CTA, one CTA per SM).
int auto_splits(int num_sms, int warps, int batch, int num_kv_heads, int max_blocks_per_seq);

// Warps per decode CTA for a layer format and GQA group size g.
int decode_warps(const tq_cache_desc& d, int g);

// Workspace layout of decode (all offsets 256-byte aligned).
struct DecodeWorkspace {
  size_t cnt_off;    // int32 [units] finished-chunk counters, at offset 0 (see kCounterRegionBytes)
  size_t qrot_off;   // fp32 [batch][Hq][d]  rotated, scaled queries (+ QJL projections)
  size_t part_off;   // fp32 [batch][Hq][splits][d] partial accumulators
  size_t ml_off;     // fp32 [batch][Hq][splits][2] (running max, denominator)
  size_t total;
};

// The counters occupy the first kCounterRegionBytes of every workspace (more only
// for shapes with more than 16384 (sequence, query head) rows).  Decode calls leave
// them at zero, so a workspace zero-filled once can serve any later call.
constexpr size_t kCounterRegionBytes = 65536;
DecodeWorkspace decode_workspace(int batch, int num_q_heads, int splits, int head_dim, bool qjl);

// One validated decode call, as the launcher sees it.
struct DecodeCall {
  const tq_cache_desc* desc;
  const void* q;
  int q_dtype;
  int batch, num_q_heads;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* ctx_lens;
  float sm_scale;
  void* out;
  int out_dtype;
  uint8_t* workspace;
  int splits;
  unsigned* status;
  bool after_append;  // enqueued right after this library's append on the same stream (tq_append_decode)
  // tq_decode_step: the new token of sequence b ([batch][H_kv][head_dim], new_dtype)
  // is written by the decode kernel itself at position context_lens[b] - 1
  const void* new_k = nullptr;
  const void* new_v = nullptr;
  int new_dtype = 0;
};

// True if the append quantizer's cell table can hold these (ascending) boundaries:
// each boundary in a cell of its own (cells are 1/63 wide on [-1, 1]).
bool cell_table_ok(const float* boundaries, int nb);

// Kernel launchers (CUDA translation units).  All enqueue on `st` and return
// the launch error, if any.
// x_v != nullptr (packed layers, which = 0): the values are quantized in the same
// launch; the caller guarantees the K and V formats agree (bits, no QJL).
// pdl: the bulk kernels (staged FWHT, tensor-core dense) are launched as programmatic
// dependents of the kernel before them and touch memory without waiting for it -- only
// for a kernel that shares no memory the launch touches (the previous layer of a
// batched append, the keys of the same append); they wait for it before completing,
// so work queued after them still finds both grids done.
cudaError_t launch_quantize(const tq_cache_desc& d, int which, const void* x, int in_dtype, const float* y,
                            const float* norms, const int64_t* slots, int64_t n_tok, unsigned* status, int num_sms,
                            cudaStream_t st, const void* x_v = nullptr, bool pdl = false);
cudaError_t launch_dequant(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n, void* out,
                           int out_dtype, unsigned* status, int num_sms, cudaStream_t st);
cudaError_t launch_decode(const DecodeCall& c, cudaStream_t st);
// Polar layers (tq_polar.cu); the generic launchers above route them here.
cudaError_t launch_polar_append(const tq_cache_desc& d, int which, const void* x, int in_dtype,
                                const int64_t* slots, int64_t n_tok, unsigned* status, int num_sms, cudaStream_t st);
cudaError_t launch_polar_dequant(const tq_cache_desc& d, int which, const int64_t* slots, int64_t n, void* out,
                                 int out_dtype, unsigned* status, int num_sms, cudaStream_t st);
cudaError_t launch_polar_decode(const DecodeCall& c, cudaStream_t st);

}  // namespace tq
