// tq_decode_attention_static: decode attention whose scratch lives inside the
// library, for callers that cannot allocate device memory themselves.
//
// Who needs it: code that runs where a device allocation is not allowed or not
// possible -- a plugin or FFI caller handed only the input and output buffers
// by a host application that owns the whole device-memory budget, or a serving
// loop that must not call cudaMalloc/cudaFree after start-up (they synchronize
// the device and can fail once the memory has been handed out).  Such callers
// cannot provide the workspace tq_decode_attention asks for.
//
// The scratch is one file-scope device array of TQ_STATIC_SCRATCH_BYTES.  Every
// GPU that loads libtq holds it until the process exits.  Host code cannot use
// the array's name as a device address, so the first call on each device looks
// the address up with cudaGetSymbolAddress (with that device current) and
// caches it; make that first call before any stream capture.  The call then
// runs the ordinary decode path with the array as its workspace.  That path
// needs the per-unit chunk counters at the start of its workspace to be zero
// when a call begins.  A __device__ array is zero-filled when the module is
// loaded, and every decode call leaves the counters it used at zero again
// (the CTA that completes a unit resets its counter; the decode kernel has no
// wait that can give up, and a call that flags a bad block id or context length
// still completes every unit), so the array never needs clearing; everything
// else in it is written before it is read within a call.  Keep the array a
// zero-initialised __device__ object for that reason.  All calls on a device
// share the one array: calls whose work overlaps on the GPU (different streams,
// or several host threads) race on it and give wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "tq_internal.h"

namespace tq {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[TQ_STATIC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxScratchDevices] = {};

// Device address of g_static_scratch on the current device (set up once per device).
tq_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxScratchDevices) return fail(TQ_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(TQ_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TQ_OK;
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_decode_attention_static(const tq_cache_desc* desc, const void* q, int q_dtype, int batch,
                                                int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                                                const int32_t* context_lens, float sm_scale, void* out, int out_dtype,
                                                int num_splits, void* stream) {
  using namespace tq;
  clear_error();
  if (batch == 0) return TQ_OK;
  if (num_splits < 0) return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention_static: num_splits < 0");
  const size_t need = tq_workspace_bytes(desc, batch, num_q_heads, max_blocks_per_seq, num_splits);
  if (need == 0) {
    tq_status s = check_desc(desc, false);
    return s != TQ_OK ? s : fail(TQ_ERR_INVALID_ARG, "tq_decode_attention_static: invalid sizes");
  }
  if (need > (size_t)TQ_STATIC_SCRATCH_BYTES)
    return fail(TQ_ERR_WORKSPACE,
                "tq_decode_attention_static: these sizes need %zu bytes of scratch but the library's static scratch "
                "holds %zu; use fewer splits, a smaller batch, or tq_decode_attention with your own workspace",
                need, (size_t)TQ_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  tq_status s = scratch_address(&scratch);
  if (s != TQ_OK) return s;
  return tq_decode_attention(desc, q, q_dtype, batch, num_q_heads, block_table, max_blocks_per_seq, context_lens,
                             sm_scale, out, out_dtype, scratch, (size_t)TQ_STATIC_SCRATCH_BYTES, num_splits, stream);
}
