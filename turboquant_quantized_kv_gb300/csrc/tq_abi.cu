// extern "C" entry points of libtq: host-side validation, the sticky device
// status word and dispatch to the kernels.  The specification of every call
// (arguments, layouts, ownership, errors) is in include/tq.h.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

// Sticky status bits set by kernels (one word per device that loads the library).
static __device__ unsigned g_tq_status;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  unsigned* status = nullptr;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

tq_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(TQ_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(TQ_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.status), g_tq_status);
    if (e != cudaSuccess) return fail(TQ_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    di.ready = true;
  }
  *out = di;
  return TQ_OK;
}

tq_status cuda_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(TQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return TQ_OK;
}

bool valid_dtype(int t) { return t == TQ_F32 || t == TQ_BF16; }

// Checks of tq_quantize_append's arguments (n_tokens == 0 passes: nothing to do).
tq_status check_append(const tq_cache_desc* desc, const void* k, const void* v, int in_dtype,
                       const int64_t* slot_mapping, int64_t n_tokens, const char* fn) {
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  if (!valid_dtype(in_dtype)) return fail(TQ_ERR_INVALID_ARG, "%s: in_dtype %d", fn, in_dtype);
  if (n_tokens < 0) return fail(TQ_ERR_INVALID_ARG, "%s: n_tokens < 0", fn);
  if (n_tokens == 0) return TQ_OK;
  if (!slot_mapping) return fail(TQ_ERR_INVALID_ARG, "%s: null slot_mapping", fn);
  if (!k && !v) return fail(TQ_ERR_INVALID_ARG, "%s: both k and v are null", fn);
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return fail(TQ_ERR_INVALID_ARG, "%s: k/v must be 16-byte aligned", fn);
  const tq_layer_format& f = desc->fmt;
  const bool packed_k = f.kv_format == TQ_KV_PACKED,
             packed_v = f.kv_format == TQ_KV_PACKED || f.kv_format == TQ_KV_K8V4;  // codebook quantizers
  if ((k && packed_k && !cell_table_ok(desc->boundaries_k, (1 << f.bits_k) - 1)) ||
      (v && packed_v && !cell_table_ok(desc->boundaries_v, (1 << f.bits_v) - 1)))
    return fail(TQ_ERR_UNSUPPORTED, "%s: codebook boundaries closer than 1/63 apart", fn);
  return TQ_OK;
}

// The launches of a checked append (n_tokens > 0): keys and values in one launch
// when their formats and tables agree.
tq_status run_append(const tq_cache_desc* desc, const void* k, const void* v, int in_dtype,
                     const int64_t* slot_mapping, int64_t n_tokens, const DeviceInfo& di, cudaStream_t st,
                     bool pdl = false) {
  const tq_layer_format& f = desc->fmt;
  const bool same_tables = std::memcmp(desc->centroids_k, desc->centroids_v, sizeof(desc->centroids_k)) == 0 &&
                           std::memcmp(desc->boundaries_k, desc->boundaries_v, sizeof(desc->boundaries_k)) == 0;
  if (k && v && f.kv_format == TQ_KV_PACKED && f.bits_k == f.bits_v && !f.qjl_k && same_tables)  // one launch
    return cuda_result(launch_quantize(*desc, 0, k, in_dtype, nullptr, nullptr, slot_mapping, n_tokens, di.status,
                                       di.num_sms, st, v, pdl),
                       "quantize K+V");
  tq_status s = TQ_OK;
  if (k) {
    s = cuda_result(launch_quantize(*desc, 0, k, in_dtype, nullptr, nullptr, slot_mapping, n_tokens, di.status,
                                    di.num_sms, st, nullptr, pdl), "quantize K");
    if (s != TQ_OK) return s;
  }
  if (v)
    s = cuda_result(launch_quantize(*desc, 1, v, in_dtype, nullptr, nullptr, slot_mapping, n_tokens, di.status,
                                    di.num_sms, st, nullptr, pdl || k != nullptr), "quantize V");
  return s;
}

// Split count of a decode call: num_splits clamped to [1, min(max_blocks, 256)], or
// the automatic choice for 0.
int resolve_splits(const tq_cache_desc* desc, int batch, int num_q_heads, int max_blocks, int num_splits) {
  if (num_splits > 0) return num_splits < max_blocks ? (num_splits > 256 ? 256 : num_splits) : (max_blocks > 256 ? 256 : max_blocks);
  return tq_auto_splits(desc, batch, num_q_heads, max_blocks);
}

// Checks of tq_decode_attention's arguments and the call they describe (batch
// == 0 passes with *c unset: nothing to do).
tq_status prepare_decode(const tq_cache_desc* desc, const void* q, int q_dtype, int batch, int num_q_heads,
                         const int32_t* block_table, int max_blocks_per_seq, const int32_t* context_lens,
                         float sm_scale, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                         int num_splits, const char* fn, DecodeCall* c) {
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  if (batch < 0) return fail(TQ_ERR_INVALID_ARG, "%s: batch < 0", fn);
  if (batch == 0) return TQ_OK;
  if (batch > 65535) return fail(TQ_ERR_UNSUPPORTED, "%s: batch %d > 65535", fn, batch);
  if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype))
    return fail(TQ_ERR_INVALID_ARG, "%s: q_dtype %d / out_dtype %d", fn, q_dtype, out_dtype);
  if (num_q_heads < 1 || num_q_heads % desc->num_kv_heads != 0)
    return fail(TQ_ERR_INVALID_ARG, "%s: num_q_heads %d not a multiple of num_kv_heads %d", fn, num_q_heads,
                desc->num_kv_heads);
  if (!q || !block_table || !context_lens || !out)
    return fail(TQ_ERR_INVALID_ARG, "%s: null q/block_table/context_lens/out", fn);
  if (max_blocks_per_seq < 1) return fail(TQ_ERR_INVALID_ARG, "%s: max_blocks_per_seq < 1", fn);
  if (num_splits < 0) return fail(TQ_ERR_INVALID_ARG, "%s: num_splits < 0", fn);
  if (!(sm_scale == sm_scale)) return fail(TQ_ERR_INVALID_ARG, "%s: sm_scale is NaN", fn);
  if (reinterpret_cast<uintptr_t>(q) & 15) return fail(TQ_ERR_INVALID_ARG, "%s: q must be 16-byte aligned", fn);
  DeviceInfo di;
  if ((s = device_info(&di)) != TQ_OK) return s;
  const int splits = resolve_splits(desc, batch, num_q_heads, max_blocks_per_seq, num_splits);
  if (splits < 1) return fail(TQ_ERR_INVALID_ARG, "%s: could not choose a split count", fn);
  const bool qjl = desc->fmt.kv_format == TQ_KV_PACKED && desc->fmt.qjl_k;
  const size_t need = decode_workspace(batch, num_q_heads, splits, desc->head_dim, qjl).total;
  if (!workspace || workspace_bytes < need)
    return fail(TQ_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", fn, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(TQ_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
  c->desc = desc;
  c->q = q;
  c->q_dtype = q_dtype;
  c->batch = batch;
  c->num_q_heads = num_q_heads;
  c->block_table = block_table;
  c->max_blocks = max_blocks_per_seq;
  c->ctx_lens = context_lens;
  c->sm_scale = sm_scale;
  c->out = out;
  c->out_dtype = out_dtype;
  c->workspace = reinterpret_cast<uint8_t*>(workspace);
  c->splits = splits;
  c->status = di.status;
  c->after_append = false;
  return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

tq_status tq_quantize_append(const tq_cache_desc* desc, const void* k, const void* v, int in_dtype,
                             const int64_t* slot_mapping, int64_t n_tokens, void* stream) {
  clear_error();
  tq_status s = check_append(desc, k, v, in_dtype, slot_mapping, n_tokens, "tq_quantize_append");
  if (s != TQ_OK || n_tokens == 0) return s;
  DeviceInfo di;
  if ((s = device_info(&di)) != TQ_OK) return s;
  return run_append(desc, k, v, in_dtype, slot_mapping, n_tokens, di, reinterpret_cast<cudaStream_t>(stream));
}

tq_status tq_quantize_append_layers(const tq_cache_desc* const* descs, int n_layers, const void* const* k,
                                    const void* const* v, int in_dtype, const int64_t* slot_mapping,
                                    int64_t n_tokens, void* stream) {
  clear_error();
  if (n_layers < 0) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_append_layers: n_layers < 0");
  if (n_layers == 0) return TQ_OK;
  if (!descs) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_append_layers: null descriptor array");
  for (int l = 0; l < n_layers; ++l) {  // every layer is checked before anything is launched
    tq_status s = check_append(descs[l], k ? k[l] : nullptr, v ? v[l] : nullptr, in_dtype, slot_mapping, n_tokens,
                               "tq_quantize_append_layers");
    if (s != TQ_OK) return s;
    for (int m = 0; m < l; ++m)
      if (descs[m]->k_cache == descs[l]->k_cache || descs[m]->v_cache == descs[l]->v_cache)
        return fail(TQ_ERR_INVALID_ARG, "tq_quantize_append_layers: layers %d and %d share a cache", m, l);
  }
  if (n_tokens == 0) return TQ_OK;
  DeviceInfo di;
  tq_status s = device_info(&di);
  if (s != TQ_OK) return s;
  for (int l = 0; l < n_layers; ++l) {
    // after the first layer: launched as programmatic dependents, without waiting for the
    // previous layer's kernel (other caches, other inputs)
    s = run_append(descs[l], k ? k[l] : nullptr, v ? v[l] : nullptr, in_dtype, slot_mapping, n_tokens, di,
                   reinterpret_cast<cudaStream_t>(stream), l > 0);
    if (s != TQ_OK) return s;
  }
  return TQ_OK;
}

tq_status tq_quantize_rotated(const tq_cache_desc* desc, int which, const float* y, const float* norms,
                              const int64_t* slot_mapping, int64_t n_tokens, void* stream) {
  clear_error();
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  if (desc->fmt.kv_format != TQ_KV_PACKED) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_rotated: packed layers only");
  if (which != 0 && which != 1) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_rotated: which %d", which);
  if (n_tokens < 0) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_rotated: n_tokens < 0");
  if (n_tokens == 0) return TQ_OK;
  if (!y || !norms || !slot_mapping) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_rotated: null pointer");
  if (reinterpret_cast<uintptr_t>(y) & 15) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_rotated: y must be 16-byte aligned");
  DeviceInfo di;
  if ((s = device_info(&di)) != TQ_OK) return s;
  return cuda_result(launch_quantize(*desc, which, nullptr, TQ_F32, y, norms, slot_mapping, n_tokens, di.status,
                                     di.num_sms, reinterpret_cast<cudaStream_t>(stream)),
                     "quantize (rotated input)");
}

int tq_auto_splits(const tq_cache_desc* desc, int batch, int num_q_heads, int max_blocks_per_seq) {
  clear_error();
  if (check_desc(desc, false) != TQ_OK || batch < 1 || num_q_heads < 1 || max_blocks_per_seq < 1) return 0;
  DeviceInfo di;
  if (device_info(&di) != TQ_OK) return 0;
  const int g = num_q_heads / desc->num_kv_heads;
  const int hpw = g <= 4 ? 4 : 8;  // heads per decode warp
  const int groups = (g + hpw - 1) / hpw;
  return auto_splits(di.num_sms, decode_warps(*desc, g), batch, desc->num_kv_heads * groups, max_blocks_per_seq);
}


size_t tq_workspace_bytes(const tq_cache_desc* desc, int batch, int num_q_heads, int max_blocks_per_seq,
                          int num_splits) {
  clear_error();
  if (check_desc(desc, false) != TQ_OK || batch < 1 || num_q_heads < 1 || max_blocks_per_seq < 1 || num_splits < 0) return 0;
  const int splits = resolve_splits(desc, batch, num_q_heads, max_blocks_per_seq, num_splits);
  if (splits < 1) return 0;
  const bool qjl = desc->fmt.kv_format == TQ_KV_PACKED && desc->fmt.qjl_k;
  return decode_workspace(batch, num_q_heads, splits, desc->head_dim, qjl).total;
}

tq_status tq_decode_attention(const tq_cache_desc* desc, const void* q, int q_dtype, int batch, int num_q_heads,
                              const int32_t* block_table, int max_blocks_per_seq, const int32_t* context_lens,
                              float sm_scale, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                              int num_splits, void* stream) {
  clear_error();
  DecodeCall c;
  tq_status s = prepare_decode(desc, q, q_dtype, batch, num_q_heads, block_table, max_blocks_per_seq, context_lens,
                               sm_scale, out, out_dtype, workspace, workspace_bytes, num_splits, "tq_decode_attention",
                               &c);
  if (s != TQ_OK || batch == 0) return s;
  return cuda_result(launch_decode(c, reinterpret_cast<cudaStream_t>(stream)), "decode attention");
}

tq_status tq_decode_step(const tq_cache_desc* desc, const void* k_new, const void* v_new, int in_dtype,
                         const void* q, int q_dtype, int batch, int num_q_heads, const int32_t* block_table,
                         int max_blocks_per_seq, const int32_t* context_lens, float sm_scale, void* out,
                         int out_dtype, void* workspace, size_t workspace_bytes, int num_splits, void* stream) {
  clear_error();
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  const tq_layer_format& f = desc->fmt;
  if (f.kv_format != TQ_KV_PACKED || f.qjl_k || f.rot_kind != TQ_ROT_HADAMARD)
    return fail(TQ_ERR_UNSUPPORTED, "tq_decode_step: packed layers with a Hadamard rotation and no QJL keys only");
  if (!valid_dtype(in_dtype)) return fail(TQ_ERR_INVALID_ARG, "tq_decode_step: in_dtype %d", in_dtype);
  if (batch > 0 && (!k_new || !v_new)) return fail(TQ_ERR_INVALID_ARG, "tq_decode_step: null k_new or v_new");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return fail(TQ_ERR_INVALID_ARG, "tq_decode_step: k_new/v_new must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(desc->rotation) & 3)
    return fail(TQ_ERR_INVALID_ARG, "tq_decode_step: rotation must be 4-byte aligned");
  DecodeCall c;
  s = prepare_decode(desc, q, q_dtype, batch, num_q_heads, block_table, max_blocks_per_seq, context_lens, sm_scale,
                     out, out_dtype, workspace, workspace_bytes, num_splits, "tq_decode_step", &c);
  if (s != TQ_OK || batch == 0) return s;
  c.new_k = k_new;
  c.new_v = v_new;
  c.new_dtype = in_dtype;
  return cuda_result(launch_decode(c, reinterpret_cast<cudaStream_t>(stream)), "decode step");
}

tq_status tq_append_decode(const tq_cache_desc* desc, const void* k, const void* v, int in_dtype,
                           const int64_t* slot_mapping, int64_t n_tokens, const void* q, int q_dtype, int batch,
                           int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* context_lens, float sm_scale, void* out, int out_dtype, void* workspace,
                           size_t workspace_bytes, int num_splits, void* stream) {
  clear_error();
  tq_status s = check_append(desc, k, v, in_dtype, slot_mapping, n_tokens, "tq_append_decode");
  if (s != TQ_OK) return s;
  DecodeCall c;
  s = prepare_decode(desc, q, q_dtype, batch, num_q_heads, block_table, max_blocks_per_seq, context_lens, sm_scale,
                     out, out_dtype, workspace, workspace_bytes, num_splits, "tq_append_decode", &c);
  if (s != TQ_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n_tokens > 0) {
    DeviceInfo di;
    if ((s = device_info(&di)) != TQ_OK) return s;
    if ((s = run_append(desc, k, v, in_dtype, slot_mapping, n_tokens, di, st)) != TQ_OK) return s;
    c.after_append = true;
  }
  if (batch == 0) return TQ_OK;
  return cuda_result(launch_decode(c, st), "decode attention");
}

tq_status tq_dequantize(const tq_cache_desc* desc, int which, const int64_t* slots, int64_t n, void* out,
                        int out_dtype, void* stream) {
  clear_error();
  tq_status s = check_desc(desc);
  if (s != TQ_OK) return s;
  if (which != 0 && which != 1) return fail(TQ_ERR_INVALID_ARG, "tq_dequantize: which %d", which);
  if (!valid_dtype(out_dtype)) return fail(TQ_ERR_INVALID_ARG, "tq_dequantize: out_dtype %d", out_dtype);
  if (n < 0) return fail(TQ_ERR_INVALID_ARG, "tq_dequantize: n < 0");
  if (n == 0) return TQ_OK;
  if (!slots || !out) return fail(TQ_ERR_INVALID_ARG, "tq_dequantize: null slots/out");
  DeviceInfo di;
  if ((s = device_info(&di)) != TQ_OK) return s;
  return cuda_result(launch_dequant(*desc, which, slots, n, out, out_dtype, di.status, di.num_sms,
                                    reinterpret_cast<cudaStream_t>(stream)),
                     "dequantize");
}

tq_status tq_get_device_status(void* stream, int32_t* code) {
  clear_error();
  if (!code) return fail(TQ_ERR_INVALID_ARG, "tq_get_device_status: null code");
  DeviceInfo di;
  tq_status s = device_info(&di);
  if (s != TQ_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if ((s = cuda_result(cudaMemcpyAsync(&v, di.status, sizeof(v), cudaMemcpyDeviceToHost, st), "read status")) != TQ_OK)
    return s;
  if ((s = cuda_result(cudaStreamSynchronize(st), "synchronize")) != TQ_OK) return s;
  if ((s = cuda_result(cudaMemsetAsync(di.status, 0, sizeof(unsigned), st), "clear status")) != TQ_OK) return s;
  if ((s = cuda_result(cudaStreamSynchronize(st), "synchronize")) != TQ_OK) return s;
  *code = (int32_t)v;
  return TQ_OK;
}

}  // extern "C"
